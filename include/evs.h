/*
 * evs.h - replay-free speculative block verification for a hybrid short-FIR /
 * modal-IIR / causal-attention target, on one GB300 (sm_103a).
 *
 * Method: "EvSpark: Lossless Speculative Decoding for Hybrid DNA Foundation Models"
 * (summary page). Figure 1(c): the target verifies the old anchor plus gamma drafts in
 * one block forward and a correction becomes the next unconsumed anchor. Figure 1(d):
 * state returns to the accepted block index k - the readable KV prefix is shortened, the
 * last L-1 outer-FIR inputs are selected and IIR state s_k is kept - with no target
 * computation replayed. Interpretation, paragraph 1: one initial-state block forward plus
 * a common state-slicing protocol (Lemma 2 block-forward contract, Lemma 3 state
 * restoration, Theorem 1 sequence-level exactness). Acceptance: greedy argmax match, or
 * rejection sampling with min(1, p/q) and a correction from norm(max(0, p - q))
 * (ReaDy summary, section 3.1 and appendix D.2).
 *
 * Target model (the pages name only the three state classes; this is the reading the
 * library implements): h = E[x]; per layer xh = h / sqrt(mean(h^2) + 1e-6), then
 *   FIR-L : v = xh W_in, y_t = sum_{j<L} taps[:, j] * v_{t-j},            h += y W_out
 *   IIR-N : u = xh W_in, s_t = lam * s_{t-1} + b * u_t (N complex poles),
 *           y = Re sum_n c_n s_{t,n},                                       h += y W_out
 *   attn  : q, k, v = xh W_q, W_k, W_v; per head softmax(q K^T / sqrt(dh)) V over the
 *           readable cache plus the block keys up to the query's position,  h += o W_o
 * logits = (h / rms(h)) W_head; p = softmax(logits / temperature).
 *
 * Conventions
 *   - Every entry point is asynchronous on the handle's stream unless stated otherwise,
 *     and never synchronises the device. Pointers marked "device" must be device memory
 *     (or managed memory) valid until the enqueued work completes.
 *   - The caller owns every buffer: weights, the workspace and all inputs and outputs.
 *     The handle stores pointers into them and owns only its host-side struct.
 *   - Matrices are "out-major": row n is output channel n, its input weights
 *     contiguous (the transpose of the math convention y = x W).
 *   - dtype EVS_DTYPE_BF16 stores weights, activations fed to projections, and K/V in
 *     bfloat16; accumulation, the residual stream, FIR inputs and the complex IIR state
 *     are fp32. EVS_DTYPE_F32 keeps everything in fp32.
 *   - Block rows are ordered m = (b * n_cand + c) * (gamma + 1) + i, i = block position
 *     (0 = anchor, i >= 1 = draft i).
 *   - Errors found on the host are returned before anything is enqueued. Kernels never
 *     trap: a condition only the device can see (a KV capacity overflow, k outside
 *     [0, gamma], a token id out of range) skips or clamps the affected access and sets a
 *     bit readable through evs_device_flags.
 */
#ifndef EVS_H
#define EVS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct evs_handle evs_handle;

typedef enum {
    EVS_OK = 0,
    EVS_ERR_INVALID_ARG = 1, /* null pointer, bad size, unsupported shape            */
    EVS_ERR_CAPACITY = 2,    /* KV rows would exceed t_max, or workspace too small   */
    EVS_ERR_STATE = 3,       /* call out of order (slice without a verify before it) */
    EVS_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed          */
} evs_status;

enum { EVS_LAYER_FIR = 0, EVS_LAYER_IIR = 1, EVS_LAYER_ATTN = 2 };
enum { EVS_DTYPE_F32 = 0, EVS_DTYPE_BF16 = 1 };
enum { EVS_MODE_GREEDY = 0, EVS_MODE_SAMPLING = 1 };
/* How several candidate blocks per sequence are verified under sampling (greedy commits
 * the candidate with the most accepted drafts under both, which is exact there):
 *   EVS_CAND_RECURSIVE   lossless: rejection sampling applied recursively across the
 *                        candidates that share the accepted prefix (a token tree with equal
 *                        prefixes merged); the output follows the target distribution.
 *   EVS_CAND_MAX_ACCEPT  each candidate tested alone with its own uniforms, the one with
 *                        the most accepted drafts committed (lowest index on ties); not
 *                        distribution-preserving in general. */
enum { EVS_CAND_RECURSIVE = 0, EVS_CAND_MAX_ACCEPT = 1 };

/* Bits of the device flag word (evs_device_flags). */
enum {
    EVS_FLAG_KV_OVERFLOW = 1u,    /* a write past t_max was skipped                     */
    EVS_FLAG_BAD_K = 2u,          /* slice saw k outside [0, gamma] or a bad candidate  */
    EVS_FLAG_EMPTY_RESIDUAL = 4u, /* max(0, p - q) summed to 0 in fp32; p was used      */
    EVS_FLAG_BAD_TOKEN = 8u,      /* a token id outside [0, vocab) was clamped          */
    EVS_FLAG_TIMEOUT = 16u        /* a kernel gave up a bounded wait; its output is void */
};

#define EVS_MAX_LAYERS 64

typedef struct {
    int32_t d;                            /* model width (multiple of 64, <= 8192)      */
    int32_t vocab;                        /* vocabulary (256 * 2^j, 256 .. 4096)        */
    int32_t n_layers;                     /* 1 .. EVS_MAX_LAYERS                        */
    int32_t layer_kind[EVS_MAX_LAYERS];   /* EVS_LAYER_*                                */
    int32_t layer_param[EVS_MAX_LAYERS];  /* FIR taps L (2..16) | IIR poles N (1,2,4,8,16,32)
                                             | attention heads H (H * head_dim == d)    */
    int32_t head_dim;                     /* attention head width (16, 32, 64 or 128)   */
    int32_t gamma;                        /* drafts per block (1..31)                   */
    int32_t batch;                        /* sequences B (1..64)                        */
    int32_t n_cand;                       /* candidate blocks C per sequence            */
    int32_t t_max;                        /* KV capacity per sequence, tokens (<= 2^21) */
    int32_t prefill_chunk;                /* tokens per sequence per prefill pass       */
    int32_t dtype;                        /* EVS_DTYPE_*                                */
    int32_t mode;                         /* EVS_MODE_*                                 */
    float temperature;                    /* p = softmax(logits / temperature), > 0     */
    float near_tie_tau;                   /* relative threshold of the near-tie flags   */
    int32_t cand_rule;                    /* EVS_CAND_* (n_cand > 1, sampling)          */
} evs_config;

typedef struct {
    const void* w_in;        /* FIR, IIR: [d][d] out-major, dtype                        */
    const void* w_out;       /* FIR, IIR: [d][d] out-major, dtype                        */
    const float* fir_taps;   /* FIR: [d][L] fp32, taps[c][j] multiplies v_{t-j}[c]        */
    const float* iir_lambda; /* IIR: [d][N][2] fp32 (re, im) poles                         */
    const float* iir_b;      /* IIR: [d][N][2] fp32 input coefficients                     */
    const float* iir_c;      /* IIR: [d][N][2] fp32 readout coefficients                   */
    const void* w_qkv;       /* attn: [3d][d] out-major, dtype; rows q (0..d-1), k, v     */
    const void* w_o;         /* attn: [d][d] out-major, dtype                              */
} evs_layer_weights;

typedef struct {
    const void* embed;                    /* [vocab][d] dtype                            */
    const void* head;                     /* [vocab][d] out-major dtype                  */
    evs_layer_weights layer[EVS_MAX_LAYERS];
} evs_weights;

/* Caller-side view of the decode state, for import / export (checkpoint and resume;
 * the slicing contract of Figure 1(d) is exactly this state). Pointers are device
 * memory except kv_len. Arrays are indexed by layer index; entries of other kinds are
 * ignored. */
typedef struct {
    int32_t* kv_len;                        /* host [B] readable KV length per sequence */
    int32_t t_stride;                       /* rows per (sequence, head) in k and v      */
    void* k[EVS_MAX_LAYERS];                /* attn: [B][H][t_stride][dh] dtype          */
    void* v[EVS_MAX_LAYERS];                /* attn: [B][H][t_stride][dh] dtype          */
    float* fir_tail[EVS_MAX_LAYERS];        /* FIR: [B][L-1][d] fp32, oldest input first */
    float* iir_state[EVS_MAX_LAYERS];       /* IIR: [B][d][N][2] fp32                    */
} evs_state_view;

/* Internal buffers exposed read-only for tests and diagnostics (evs_debug_buffer). */
enum {
    EVS_BUF_LOGITS = 0,     /* [B*C*(gamma+1)][vocab] fp32, last verify                 */
    EVS_BUF_FIR_STAGE = 1,  /* layer: [B][C][L-1+gamma+1][d] fp32 = [tail || inputs v]    */
    EVS_BUF_IIR_U = 2,      /* layer: [B][C][gamma+1][d] fp32 scan inputs u_0..u_gamma    */
    EVS_BUF_K_CACHE = 3,    /* layer: [B][H][t_max][dh] dtype                             */
    EVS_BUF_V_CACHE = 4,    /* layer: [B][H][t_max][dh] dtype                             */
    EVS_BUF_K_SIDE = 5,     /* layer, n_cand > 1: [B][C][H][gamma+1][dh] dtype block keys  */
    EVS_BUF_V_SIDE = 6,     /* layer, n_cand > 1: [B][C][H][gamma+1][dh] dtype             */
    EVS_BUF_KV_LEN = 7,     /* [B] int32                                                  */
    EVS_BUF_FIR_TAIL = 8,   /* layer: [B][L-1][d] fp32                                    */
    EVS_BUF_IIR_STATE = 9,  /* layer: [B][d][N][2] fp32                                   */
    EVS_BUF_CAND_K = 10,    /* [B][C] int32 accepted drafts per candidate, last verify
                               (EVS_CAND_RECURSIVE sampling: drafts on the accepted path) */
    EVS_BUF_CAND_CORR = 11  /* [B][C] int32 correction per candidate, last verify
                               (EVS_CAND_RECURSIVE sampling: -1 but for the committed one) */
};

typedef struct {
    void* ptr;        /* device pointer into the workspace (do not write)              */
    size_t bytes;
} evs_buffer_info;

/* Bytes of device workspace that evs_create needs for this configuration (0 if the
 * configuration is invalid). Pure host function. */
size_t evs_workspace_bytes(const evs_config* cfg);

/* Validate the configuration, lay out state and scratch buffers inside the caller's
 * workspace (device, >= evs_workspace_bytes, 256-byte aligned) and build the handle.
 * Weights are device pointers in the layouts above and must outlive the handle.
 * stream is a cudaStream_t (NULL = legacy default stream). The state starts empty
 * (kv_len = 0, FIR tails and IIR states zero); the zeroing is enqueued on the stream.
 * Returns EVS_ERR_INVALID_ARG for a bad configuration or pointer, EVS_ERR_CAPACITY if
 * ws_bytes is too small, EVS_ERR_CUDA if a CUDA call fails. */
evs_status evs_create(const evs_config* cfg, const evs_weights* weights, void* workspace,
                      size_t ws_bytes, void* stream, evs_handle** out);

/* Free the host-side handle. Does not touch caller-owned memory. NULL is allowed. */
void evs_destroy(evs_handle* h);

/* Change the stream later calls enqueue on (a cudaStream_t). */
evs_status evs_set_stream(evs_handle* h, void* stream);

/* Return the state to empty (kv_len 0, zero FIR tails and IIR states). */
evs_status evs_reset(evs_handle* h);

/* Consume P prefix tokens per sequence from the current state, prefill_chunk tokens per
 * pass, committing every pass (no logits are produced). tokens: device int32 [B][P],
 * ids in [0, vocab). Prefill is excluded from the pages' token benchmarks (Perspective,
 * paragraph 1). EVS_ERR_CAPACITY if kv_len + P could exceed t_max. */
evs_status evs_prefill(evs_handle* h, const int32_t* tokens, int32_t P);

/* One block forward plus acceptance (Figure 1(c); Lemma 2).
 *   tokens   device int32 [B][C][gamma+1]: position 0 is the anchor, 1..gamma drafts.
 *   anchor   device int32 [B] or NULL: when given, replaces tokens[b][c][0] for every
 *            candidate (pass the previous round's correction to chain rounds).
 *   q_probs  device fp32 [B][C][gamma][vocab]: draft distributions (sampling mode; NULL
 *            in greedy mode).
 *   uniforms device fp32 [B][C][gamma+1] in [0, 1): u[j] tests draft j+1 by
 *            u * q(d) < p(d); u[gamma] draws the correction or bonus by inverse CDF over
 *            ascending ids (sampling mode; NULL in greedy mode).
 * Outputs (device, written by the enqueued kernels):
 *   accepted_len [B] int32: k, accepted drafts of the committed candidate (0..gamma).
 *   correction   [B] int32: next anchor (correction at the first rejection, or bonus).
 *   best_cand    [B] int32 or NULL: committed candidate (see EVS_CAND_*: the lowest
 *                candidate on the accepted path, or the most accepted drafts with the
 *                lowest index on ties); required when n_cand > 1.
 *   near_tie     [B] uint32 or NULL: 1 when a decision was within near_tie_tau of
 *                flipping (greedy top-2 logit gap < tau * rms(logits); |u q - p| < tau p;
 *                u * sum(r) within tau * sum(r) of an inverse-CDF boundary).
 * Writes the block's K/V rows, FIR inputs and IIR scan inputs u_0..u_gamma into the
 * workspace for evs_slice_state. State itself is not modified.
 * EVS_ERR_CAPACITY if kv_len + gamma + 1 could exceed t_max. */
evs_status evs_verify_block(evs_handle* h, const int32_t* tokens, const int32_t* anchor,
                            const float* q_probs, const float* uniforms,
                            int32_t* accepted_len, int32_t* correction, int32_t* best_cand,
                            uint32_t* near_tie);

/* State slicing at the accepted index (Figure 1(d); Lemma 3), in place, no replay of the
 * forward: kv_len += k + 1 (for n_cand > 1 the chosen candidate's k+1 block K/V rows are
 * first copied into the cache), FIR tail <- the last L-1 inputs up to block position k, IIR
 * state <- s_k (k+1 steps of the diagonal recurrence from the pre-round state over the kept
 * scan inputs, the same operations as the verify's scan). accepted_len and best_cand are
 * device int32 [B] (usually the outputs of the verify; best_cand may be NULL when
 * n_cand == 1). k stays on the device: nothing is read back. EVS_ERR_STATE if no verify was
 * enqueued since the last slice, prefill, decode step or import. */
evs_status evs_slice_state(evs_handle* h, const int32_t* accepted_len, const int32_t* best_cand);

/* Replay-based recovery, the ablation that slicing replaces (EvSpark summary,
 * Interpretation: slicing against a second target forward over the accepted prefix). After
 * evs_verify_block, k and the committed candidate are read back to the host (the stream is
 * synchronised), then a committed forward runs over that candidate's accepted tokens
 * [anchor, d_1..d_k] from the pre-round state, as a prefill does. The state it leaves equals
 * the one evs_slice_state leaves, up to rounding. One sequence only (batch == 1): the
 * accepted lengths of different sequences differ.
 *   tokens, anchor  as given to the verify (anchor may be NULL).
 *   accepted_len, best_cand  the verify's outputs (device; best_cand NULL when n_cand == 1).
 * EVS_ERR_STATE without a preceding verify; EVS_ERR_INVALID_ARG if batch > 1, a pointer is
 * missing, or k / the candidate read back is out of range. */
evs_status evs_replay_state(evs_handle* h, const int32_t* tokens, const int32_t* anchor,
                            const int32_t* accepted_len, const int32_t* best_cand);

/* One step of plain autoregressive decoding: the target's native token-by-token loop that
 * block verification is measured against (EvSpark summary, Interpretation: the
 * identity-drafter control is reported as a multiple of native throughput). Every
 * sequence consumes one token and its state advances in place (the K/V row is appended,
 * the FIR tail shifts, the IIR state takes one step), then the next token is drawn from
 * softmax(logits / temperature) of the new position: the argmax, lowest id on ties
 * (greedy mode), or the inverse CDF at u[b] over ascending ids (sampling mode). Uses the
 * verify's kernels with one row per sequence.
 *   tokens    device int32 [B]: the token each sequence consumes.
 *   uniforms  device fp32 [B] in [0, 1) (sampling mode; NULL in greedy mode).
 *   next      device int32 [B]: the drawn next token. It may alias tokens (the draw is
 *             written after every read of tokens, in stream order).
 *   near_tie  device uint32 [B] or NULL: 1 when the draw was within near_tie_tau of
 *             flipping (same tests as evs_verify_block).
 * The step's logits are left in EVS_BUF_LOGITS rows [0, B). EVS_ERR_INVALID_ARG for a
 * missing pointer, EVS_ERR_CAPACITY if kv_len + 1 could exceed t_max. */
evs_status evs_decode_step(evs_handle* h, const int32_t* tokens, const float* uniforms, int32_t* next,
                           uint32_t* near_tie);

/* Copy a caller state into the handle (import) or the handle's state out (export).
 * Enqueued copies; export writes kv_len to the host view after synchronising the
 * stream. Import rejects kv_len > t_max or > t_stride with EVS_ERR_CAPACITY. */
evs_status evs_import_state(evs_handle* h, const evs_state_view* view);
evs_status evs_export_state(evs_handle* h, const evs_state_view* view);

/* Read-only location of an internal buffer (see EVS_BUF_*); layer is a layer index
 * where the buffer is per layer. EVS_ERR_INVALID_ARG if the buffer does not exist. */
evs_status evs_debug_buffer(evs_handle* h, int32_t which, int32_t layer, evs_buffer_info* out);

/* Synchronise the stream and return the device flag word (EVS_FLAG_*); clear it when
 * clear != 0. */
evs_status evs_device_flags(evs_handle* h, uint32_t* flags, int32_t clear);

/* Kernel kinds for per-kind timing. */
enum {
    EVS_K_EMBED = 0, EVS_K_NORM = 1, EVS_K_GEMM = 2, EVS_K_FIR = 3, EVS_K_IIR = 4,
    EVS_K_KV_WRITE = 5, EVS_K_ATTN = 6, EVS_K_ATTN_COMBINE = 7, EVS_K_ACCEPT = 8,
    EVS_K_SLICE = 9, EVS_K_ADVANCE = 10, EVS_K_COUNT = 11
};

/* Per-kernel-kind timing with CUDA events (tracing for measurement; the pages describe no
 * tracing mechanism). While enabled, every launch is bracketed by two events recorded on
 * the handle's stream, so calls must not be captured into a CUDA graph. evs_profile_read
 * synchronises the stream and returns, for each kind < n, the launches and summed
 * milliseconds since the previous read, then clears the counters. */
evs_status evs_profile_enable(evs_handle* h, int32_t on);
evs_status evs_profile_read(evs_handle* h, int32_t* launches, float* ms, int32_t n);

/* Number of kernel launches the last public call enqueued (for accounting). */
int32_t evs_last_launch_count(evs_handle* h);

/* Diagnostics: Y[m][n] (+)= sum_k X[m][k] W[n][k] with the library's projection kernel
 * (the same launch path the block forward uses). X: device bf16 [x_rows][K] (x_rows >= M),
 * W: device bf16 out-major [N][K], Y: device fp32 [M][ldy]. Uses the handle's stream and
 * split-K scratch; needs a bf16 handle, M <= 512, N % 128 == 0, K % 64 == 0, K <= d and
 * N <= max(3d, vocab). EVS_ERR_INVALID_ARG otherwise. */
evs_status evs_debug_projection(evs_handle* h, const void* X, int32_t x_rows, const void* W, float* Y,
                                int32_t M, int32_t N, int32_t K, int32_t ldy, int32_t accumulate);

/* Projection for callers that cannot allocate device memory: no handle, no workspace,
 * no cudaMalloc / cudaFree or allocating library call. The pages have no counterpart of
 * this entry point; it exists for hosts that own all device memory and forbid allocation
 * while they execute (plugin-style engines), and for latency-critical loops where an
 * allocation would synchronise the device.
 * Computes Y[m][n] (+)= sum_k X[m][k] W[n][k] with the same tcgen05 kernel as
 * evs_debug_projection; split-K partial sums always go through the fixed array (never
 * through a thread-block cluster). X: device bf16 [x_rows][K] (x_rows >= M); W: device bf16
 * out-major [N][K]; Y: device fp32 [M][ldy]; stream: a cudaStream_t. Needs M <= 512,
 * N % 128 == 0, K % 64 == 0.
 * Scratch: one fixed array of 8 MiB of fp32 partial sums, 256 arrival counters and a flag
 * word, compiled into the library and held on every GPU that loads it until the process
 * exits. The K split is capped so that its partial sums (splits x M x N floats) fit 2^21
 * floats (a shape that fits no split runs unsplit), so the only size limit is N <= 32768
 * (one counter per 128-channel tile); wider N returns EVS_ERR_CAPACITY.
 * The first call on a device (of this function or evs_projection_noalloc_flags) looks up
 * the array's device address, sets the kernel's shared-memory limit for that device and
 * clears the flag word; make that first call before any stream capture. The set-up is
 * guarded, so host threads may make their first calls concurrently. A device reset
 * (cudaDeviceReset) invalidates it: reload the library after one.
 * Every call reuses the same array and finds the previous call's contents there; the
 * counters are cleared on the stream at each call. Calls that overlap on the GPU (issued
 * on different streams, or from several host threads) race on it: order them on one
 * stream. A kernel that gives up a bounded wait sets EVS_FLAG_TIMEOUT in the array's flag
 * word, and Y is then void; read the word with evs_projection_noalloc_flags.
 * EVS_ERR_INVALID_ARG for bad shapes or pointers, EVS_ERR_CUDA if a CUDA call fails. */
evs_status evs_projection_noalloc(const void* X, int32_t x_rows, const void* W, float* Y, int32_t M,
                                  int32_t N, int32_t K, int32_t ldy, int32_t accumulate, void* stream);

/* Device status of evs_projection_noalloc on the current device: synchronises stream, then
 * writes to *flags the EVS_FLAG_* bits (EVS_FLAG_TIMEOUT) that its calls have set since the
 * word was last cleared, and clears it when clear != 0 (enqueued on stream). Allocates
 * nothing. EVS_ERR_INVALID_ARG for a null flags pointer, EVS_ERR_CUDA if a CUDA call
 * fails. */
evs_status evs_projection_noalloc_flags(uint32_t* flags, int32_t clear, void* stream);

/* Static description of a status code. */
const char* evs_status_str(evs_status s);

#ifdef __cplusplus
}
#endif
#endif /* EVS_H */
