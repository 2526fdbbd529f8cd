// Internal layout of a handle and the kernel launchers it drives.
#pragma once

#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/evs.h"

namespace evs {

// Per-layer device pointers, also mirrored into device memory for the slice kernel.
struct LayerDesc {
    int32_t kind, param;           // EVS_LAYER_*, L | N | H
    float* tail;                   // FIR [B][L-1][d]
    float* stage;                  // FIR [B][C][L-1+T][d]
    float2* state;                 // IIR [B][d][N]
    float* uin;                    // IIR [B][C][T][d]: the verify pass's scan inputs u_t
    const float2* lam;             // IIR [d][N] poles and input weights (the slice kernel
    const float2* bq;              // recomputes s_k from the state and u_0..u_k)
    void* kc;                      // attn [B][H][t_max][dh]
    void* vc;
    void* ks;                      // attn, C > 1: [B][C][H][T][dh]
    void* vs;
};

struct Geometry {
    int B, C, T;      // verify: T = gamma + 1
    int M_verify;     // B*C*T
    int M_max;        // max(M_verify, B*prefill_chunk)
    int q_max;        // max queries per sequence in a pass (C*T or prefill_chunk)
    int h_max;        // max attention heads over layers
    int kv_chunk;     // prefix keys per attention split
    int kv_splits;    // ceil(t_max / kv_chunk)
};

// Prefix chunking of the tensor-core attention for one pass shape (attn_fa.cu).
struct AttnPlan {
    int ok;          // 1 if the tensor-core kernel takes this pass
    int runs;        // 1: persistent grid over runs of key tiles; 0: one CTA per chunk
    int n_q;         // query rows of the products (128, padded)
    int tiles;       // most 128-key tiles a CTA streams
    int splits;      // chunks of the prefix per sequence and head
    int stages;      // TMA ring depth (32 KiB stages)
    int ncols;       // TMEM columns
    int smem;        // dynamic shared memory bytes
};

// Fused-norm extras of one projection (null members are unused).
struct Pass;
struct GemmFuse {
    const float* ssq_in;     // rows scaled by 1/rms from these per-tile sums of squares
    int ssq_tiles, ssq_ld, norm_d;
    __nv_bfloat16* hb_out;   // bf16 copy of the final values
    int hb_ld;
    float* ssq_out;          // per-tile sums of squares of the final values
    int mix_layer;           // >= 0: run this FIR / IIR layer's mixer in the epilogue if it fits
    int kv_layer;            // >= 0: write this attention layer's K/V from the epilogue
    const Pass* pass;        // the pass shape (needed by the two above)
};

// A pass runs B sequences x C candidates x T block positions; row m = (b*C + c)*T + i.
struct Pass {
    int B, C, T;        // sequences, candidates, positions per candidate
    int M;              // B*C*T
    int commit;         // 1: prefill pass, state updated in place (C == 1)
    int kv_in_cache;    // 1: block K/V rows go to cache rows kv_base[b] + i (C == 1)
};

}  // namespace evs

struct evs_handle {
    evs_config cfg;
    evs_weights w;
    cudaStream_t stream;
    char* ws;
    size_t ws_bytes;
    evs::Geometry g;
    // control words (device)
    int32_t* kv_len;      // [B]
    int32_t* kv_base;     // [B] readable length at the start of the current pass
    uint32_t* flags;      // [1]
    int32_t* cand_k;      // [B*C]
    int32_t* cand_corr;   // [B*C]
    uint32_t* cand_tie;   // [B*C]
    // activations (device)
    float* h;             // [M_max][d] residual stream
    void* act;            // [M_max][d] dtype: normalised input or mixer output
    float* y;             // [M_max][3d] projection outputs
    float* logits;        // [M_verify][vocab]
    float* attn_part;     // [B][H_max][splits][q_max][dh + 2]
    int fused;            // norm folded into the projections (bf16, all shapes on tcgen05)
    __nv_bfloat16* hb;    // [M_max][d] bf16 copy of the residual stream (fused path)
    float* ssq;           // [d / 128][M_max] per-tile sums of squares of h (fused path)
    float* gemm_part;     // split-K partial sums fp32
    size_t gemm_part_floats;
    int* gemm_counters;   // [max(3d, vocab) / 128] split-K arrival counters
    int tc_smem_max;      // dynamic shared memory the projection kernel may use (bytes)
    evs::AttnPlan plan_verify, plan_prefill;   // tensor-core attention chunking per pass
    evs::LayerDesc layer[EVS_MAX_LAYERS];
    evs::LayerDesc* layer_dev;   // device copy
    // sizes of per-layer buffers (bytes), for evs_debug_buffer
    size_t stage_bytes[EVS_MAX_LAYERS], uin_bytes[EVS_MAX_LAYERS], cache_bytes[EVS_MAX_LAYERS],
        side_bytes[EVS_MAX_LAYERS], tail_bytes[EVS_MAX_LAYERS], state_bytes[EVS_MAX_LAYERS];
    // host bookkeeping
    long long kv_hi;      // host upper bound of max_b kv_len
    int verified;         // a verify was enqueued since the last slice / prefill
    int launches;         // kernels enqueued by the last public call
    int pdl;              // launch with programmatic dependent launch
    int fuse_mixer;       // run FIR / IIR mixers in the in-projection epilogue when they fit
    void* prof;           // evs::Profiler*, lazily created
    int prof_on;
};

namespace evs {

// ---- per-kind event timing (evs_api.cu) --------------------------------------------------
void prof_begin(evs_handle* h, int kind);
void prof_end(evs_handle* h, int kind);

// ---- kernel launchers (kernels.cu) --------------------------------------------------------
void launch_embed(evs_handle* h, const int32_t* tokens, int tok_stride_bc, const int32_t* anchor,
                  const Pass& p);
void launch_rmsnorm(evs_handle* h, const Pass& p);
// fused (if non-null) returns bit 0: the mixer ran in the epilogue, bit 1: K/V were written
void launch_gemm(evs_handle* h, const void* A, const void* W, float* Y, int M, int N, int K,
                 int ldy, int accumulate, const GemmFuse* fz = nullptr, int* fused = nullptr);
// tcgen05 projection (gemm_tc.cu); false when it cannot take the shape
bool gemm_tc_supported(int M, int N, int K);
int gemm_tc_init();
int tc_cta_target();
// tcgen05 attention (attn_fa.cu): a persistent grid of kAttnGrid CTAs
constexpr int kAttnGrid = 152;
AttnPlan attn_plan(int Q, int B, int H, int t_max, int smem_max);
int attn_init();
bool launch_attn_tensor(evs_handle* h, int layer, const Pass& p, const AttnPlan& plan);
// 3-D tensor map over a [bh][t_max][128] bf16 K or V cache, boxes of 128 rows x 64 columns
bool make_kv_map(CUtensorMap* m, const void* base, int t_max, int bh);
bool launch_gemm_tc(evs_handle* h, const void* X, int x_rows, const void* W, float* Y, int M, int N,
                    int K, int ldy, int accumulate, const GemmFuse* fz = nullptr, int* fused = nullptr);
void launch_fir(evs_handle* h, int layer, const Pass& p);
void launch_iir(evs_handle* h, int layer, const Pass& p, const float* u, int ldu);
void launch_kv_write(evs_handle* h, int layer, const Pass& p);
void launch_attention(evs_handle* h, int layer, const Pass& p);
void launch_accept(evs_handle* h, const int32_t* tokens, const float* q, const float* u,
                   int32_t* acc, int32_t* corr, int32_t* cand, uint32_t* tie);
void launch_slice(evs_handle* h, const int32_t* k, const int32_t* cand);
void launch_pick(evs_handle* h, const float* u, int32_t* next, uint32_t* tie);
void launch_advance(evs_handle* h, int T);

}  // namespace evs
