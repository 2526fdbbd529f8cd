// Split-KV attention over the readable KV prefix for up to 128 queries per sequence (every
// block position of every candidate, or a prefill chunk), streamed through tcgen05 tensor
// cores with an online softmax.
//
// Work: the key tiles of every (sequence, head) prefix laid end to end, worked out from the
// prefix lengths at run time. Either one CTA per (chunk, sequence x head), a chunk being an
// equal share of that prefix's tiles, or (when that would take many waves) a persistent grid
// of one CTA per SM taking equal runs of tiles, a run possibly crossing from one (sequence,
// head) into the next; each segment of a run is a chunk with its own partials. The queries
// are the 128 rows (TMEM lanes) of every product, padded with zero rows:
//   S[q][key]  = Q . K_t^T        (A = Q, K-major; B = K tile, K-major; D in TMEM, two buffers)
//   P          = exp2(S*scale*log2e - m)   one thread per query row, in bf16 to shared memory
//   O[q][dh]  += P . V_t          (A = P, K-major; B = V tile read MN-major; D in TMEM)
// The running maximum m of a row moves only when a tile's maximum exceeds it by more than
// 2^8 in the exponent (the stored exponentials stay below 256 otherwise); then the thread
// rescales its row of O and of the running sum l first. The CTA writes the unnormalised
// partials (o, m, l) per query in the layout the combine kernel merges.
//
// Pipeline: K runs one tile ahead of V in the TMA ring (K0, K1, V0, K2, V1, ...), so the
// score product of tile t+1 runs while the softmax of tile t does; P is double-buffered.
// Warps 0-7 stage Q, run the softmax and the epilogue: warp w owns TMEM lanes
// 32(w%4)..32(w%4)+31 (query rows) and keys 64(w/4)..64(w/4)+63 of every tile, the two warps
// of a row group agreeing on the row maximum through shared memory; warps whose rows are all
// padding sit out. Warp 8 drives TMA and allocates TMEM, warp 9 issues the MMAs. dh = 128.
#include <cudaTypedefs.h>
#include <math.h>

#include "evs_common.cuh"
#include "sm100_ptx.cuh"

namespace evs {

constexpr int FA_ROWS = 128;                  // query rows per CTA (MMA M)
constexpr int FA_KEYS = 128;                  // keys per tile
constexpr int FA_DH = 128;
constexpr int FA_TILE = FA_KEYS * FA_DH * 2;  // 32 KiB: two 64-column swizzled halves
constexpr int FA_HALF = FA_TILE / 2;
constexpr int FA_THREADS = 320;
constexpr float FA_RESCALE_LOG2 = 8.f;        // lazy rescale threshold (exponent of 2)
constexpr int FA_MAX_B = 512;                 // sequences a launch can hold
constexpr int FA_GRID = kAttnGrid;            // persistent CTAs: one per SM

struct FaArgs {
    const float* y;        // projection output, q in columns [head*dh, head*dh + dh)
    int ldy, B, H, Q;      // sequences, heads, queries per sequence (<= 128)
    int splits, q_stride, stages;   // splits: partial slots per (sequence, head)
    float scale;
    const int32_t* kv_base;
    float* part;           // [B][H][splits][q_stride][dh + 2]
    uint32_t* flags;
};

__device__ __forceinline__ uint32_t fa_sw128(int row, int chunk16) {
    // byte offset of 16-byte chunk chunk16 (0..7) of row `row` in a [rows][64] bf16 block
    // with the 128-byte swizzle
    return (uint32_t)row * 128u + ((uint32_t)(chunk16 ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Position `pos` of the run of every (sequence, head)'s key tiles, laid end to end (sequence
// major): its (sequence, head), tile within that prefix, and where that prefix starts.
// nt[b] = key tiles of sequence b.
__device__ __forceinline__ void fa_locate(const int* nt, int B, int H, int pos, int& bh, int& t, int& start,
                                          int& ntb) {
    int base = 0;
    bh = 0;
    t = 0;
    start = 0;
    ntb = 1;
    for (int b = 0; b < B; ++b) {
        const int span = H * nt[b];
        if (pos < base + span) {
            const int h = (pos - base) / nt[b];
            t = (pos - base) - h * nt[b];
            bh = b * H + h;
            start = base + h * nt[b];
            ntb = nt[b];
            return;
        }
        base += span;
    }
}

template <bool RUNS>
__global__ void __launch_bounds__(FA_THREADS, 1)
attn_fa_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, FaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot[1];
    __shared__ volatile int abort_flag[1];
    __shared__ float xmax[2][2][FA_ROWS];   // [tile parity][key half]: a tile's row maxima
    __shared__ float xsum[FA_ROWS];      // the second half's running sums, for the epilogue

    __shared__ int nt_s[RUNS ? FA_MAX_B : 1];   // key tiles of each sequence's readable prefix
    __shared__ int n_s[RUNS ? FA_MAX_B : 1];    // its length in keys

    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // This CTA's tiles [lo, hi): with runs, a range of the key tiles of every (sequence, head)
    // laid end to end; with chunks, tile indices within the prefix of (sequence, head) bh0.
    int lo, hi, W = 1, bh0 = 0, n0 = 0;
    if constexpr (RUNS) {
        for (int b = tid; b < a.B; b += blockDim.x) {
            n_s[b] = a.kv_base[b];
            nt_s[b] = (n_s[b] + FA_KEYS - 1) / FA_KEYS;
        }
        __syncthreads();
        int total = 0;
        for (int b = 0; b < a.B; ++b) total += a.H * nt_s[b];
        W = (total + (int)gridDim.x - 1) / (int)gridDim.x;
        lo = W * (int)blockIdx.x;
        hi = min(lo + W, total);
    } else {   // one chunk: an equal share of the key tiles of prefix (sequence, head) blockIdx.y
        bh0 = blockIdx.y;
        const int split = blockIdx.x;
        n0 = a.kv_base[bh0 / a.H];
        const int nt = (n0 + FA_KEYS - 1) / FA_KEYS;
        lo = (int)((long long)nt * split / a.splits);
        hi = (int)((long long)nt * (split + 1) / a.splits);
        if (lo >= hi) {   // share past the readable prefix: empty partial
            float* part = a.part + ((size_t)bh0 * a.splits + split) * a.q_stride * (FA_DH + 2);
            for (int i = tid; i < a.Q; i += blockDim.x) {
                part[(size_t)i * (FA_DH + 2) + FA_DH] = -INFINITY;
                part[(size_t)i * (FA_DH + 2) + FA_DH + 1] = 0.f;
            }
            return;
        }
    }
    if (lo >= hi) return;                                        // no work for this CTA

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = smem;                                   // [2 halves][128][128 B]
    uint8_t* sP = sQ + FA_TILE;                           // [2 buffers][2 halves][128][128 B]
    uint8_t* ring = sP + 2 * FA_TILE;                     // [stages][2 halves][128][128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)a.stages * FA_TILE);
    uint64_t* empty = full + a.stages;
    uint64_t* s_full = empty + a.stages;                  // [2] scores of a tile in TMEM
    uint64_t* p_full = s_full + 2;                        // [2] P of a tile in shared memory
    uint64_t* pv_done = p_full + 2;                       // [2] P.V of a tile complete
    uint64_t* drain = pv_done + 2;                        // every MMA of the CTA complete
    uint64_t* q_ready = drain + 1;                        // Q of the next segment staged
    int issued = 0;                                       // TMA steps issued (warp 8, lane 0)
    const int quarters = (a.Q + 31) / 32;                 // row groups holding real queries

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 2 * quarters);   // one arrival per working softmax warp
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(drain, 1);
        mbar_init(q_ready, 2 * quarters);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // The segments of this CTA's tiles, identical in every role: (sequence x head, first
    // tile, tile count, partial slot).
    auto segment = [&](int pos, int& bh, int& t0, int& ntiles, int& slot) {
        if constexpr (RUNS) {
            int start, ntb;
            fa_locate(nt_s, a.B, a.H, pos, bh, t0, start, ntb);
            ntiles = min(ntb - t0, hi - pos);
            slot = (int)blockIdx.x - start / W;
        } else {
            bh = bh0;
            t0 = pos;
            ntiles = hi - pos;
            slot = blockIdx.x;
        }
    };
    // stage Q rows (fp32 -> bf16, swizzled K-major) of (sequence x head) bh: row r, dims
    // 64g..64g+63, zero past Q
    auto stage_q = [&](int bh, int r, int g) {
        const int b = bh / a.H, head = bh % a.H;
        const float* qrow = a.y + ((size_t)b * a.Q + r) * a.ldy + (size_t)head * FA_DH + g * 64;
#pragma unroll 4
        for (int c = 0; c < 8; ++c) {   // 8 chunks of 8 dims
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (r < a.Q) {
                const float4 x0 = *reinterpret_cast<const float4*>(qrow + c * 8);
                const float4 x1 = *reinterpret_cast<const float4*>(qrow + c * 8 + 4);
                u.x = pack_bf16x2(x0.x, x0.y);
                u.y = pack_bf16x2(x0.z, x0.w);
                u.z = pack_bf16x2(x1.x, x1.y);
                u.w = pack_bf16x2(x1.z, x1.w);
            }
            *reinterpret_cast<uint4*>(sQ + (size_t)g * FA_HALF + fa_sw128(r, c)) = u;
        }
        fence_proxy_async_smem();
    };
    if (warp < 8) {   // the first segment's Q by every row group (padding rows zero for good)
        int bh, t0, nts, slot;
        segment(lo, bh, t0, nts, slot);
        stage_q(bh, (warp & 3) * 32 + lane, warp >> 2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t o_col = 256;                            // S buffers at columns 0 and 128

    if (warp == 8) {
        if (lane == 0) {  // ---- TMA: per segment K0, K1, V0, K2, V1, ..., V_{n-1} -----------------
            const uint64_t pol = policy_evict_first();
            int i = 0;     // ring step over all segments
            bool ok = true;
            for (int pos = lo; pos < hi && ok;) {
                int bh, t0, ntiles, slot;
                segment(pos, bh, t0, ntiles, slot);
                const int steps = 2 * ntiles;
                for (int j = 0; j < steps; ++j, ++i) {
                    const int s = i % a.stages;
                    const uint32_t ph = (uint32_t)(i / a.stages) & 1u;
                    if (i >= a.stages && !mbar_wait(&empty[s], ph ^ 1u)) { *abort_flag = 1; ok = false; break; }
                    bool is_k;
                    int t;
                    if (j == 0) { is_k = true; t = 0; }
                    else if (j == steps - 1) { is_k = false; t = ntiles - 1; }
                    else if (j & 1) { is_k = true; t = (j + 1) >> 1; }
                    else { is_k = false; t = (j >> 1) - 1; }
                    const int row = (t0 + t) * FA_KEYS;
                    uint8_t* dst = ring + (size_t)s * FA_TILE;
                    mbar_arrive_expect_tx(&full[s], (uint32_t)FA_TILE);
                    tma_load_3d(dst, is_k ? &tmK : &tmV, 0, row, bh, &full[s], pol);
                    tma_load_3d(dst + FA_HALF, is_k ? &tmK : &tmV, 64, row, bh, &full[s], pol);
                    issued = i + 1;
                }
                pos += ntiles;
                if constexpr (!RUNS) break;
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        if (lane == 0) {  // ---- MMA issuer ----------------------------------------------------
            const uint32_t id_s = idesc_bf16_f32(FA_ROWS, FA_KEYS);
            const uint32_t id_o = idesc_bf16_f32_bmn(FA_ROWS, FA_DH);
            const uint32_t q0 = smem_u32(sQ);
            bool ok = true;
            int i = 0;    // ring step over all segments
            int gt0 = 0;  // tiles of earlier segments (buffer and phase parity run on)
            auto score = [&](int gt) {         // S[gt & 1] = Q . K^T
                const int s = i % a.stages;
                if (!mbar_wait(&full[s], (uint32_t)(i / a.stages) & 1u)) { ok = false; return; }
                tc_fence_after();
                const uint32_t k0 = smem_u32(ring + (size_t)s * FA_TILE);
#pragma unroll
                for (int kk = 0; kk < FA_DH / 16; ++kk) {
                    const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32u;
                    tc_mma_f16(tmem + (uint32_t)(gt & 1) * 128u, smem_desc_sw128(q0 + half * FA_HALF + off),
                               smem_desc_sw128(k0 + half * FA_HALF + off), id_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&empty[s]);
                tc_commit(&s_full[gt & 1]);
                ++i;
            };
            auto pv = [&](int gt, bool first) {   // O (+)= P . V
                if (!mbar_wait(&p_full[gt & 1], (uint32_t)(gt >> 1) & 1u)) { ok = false; return; }
                const int s = i % a.stages;
                if (!mbar_wait(&full[s], (uint32_t)(i / a.stages) & 1u)) { ok = false; return; }
                tc_fence_after();
                const uint32_t v0 = smem_u32(ring + (size_t)s * FA_TILE);
                const uint32_t p0 = smem_u32(sP + (size_t)(gt & 1) * FA_TILE);
#pragma unroll
                for (int kk = 0; kk < FA_KEYS / 16; ++kk) {
                    const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32u;
                    tc_mma_f16(tmem + o_col, smem_desc_sw128(p0 + half * FA_HALF + off),
                               smem_desc_sw128_mn(v0 + (uint32_t)kk * 16u * 128u, FA_HALF), id_o,
                               (!first || kk > 0) ? 1u : 0u);
                }
                tc_commit(&empty[s]);
                tc_commit(&pv_done[gt & 1]);
                ++i;
            };
            int seg = 0;
            for (int pos = lo; pos < hi && ok; ++seg) {
                int bh, t0, ntiles, slot;
                segment(pos, bh, t0, ntiles, slot);
                // a later segment's Q staged (after the previous segment's last P.V, so sQ is
                // free); the first one was staged before the CTA-wide barrier
                if (seg > 0) {
                    if (!mbar_wait(q_ready, (uint32_t)(seg - 1) & 1u)) { ok = false; break; }
                    tc_fence_after();
                }
                score(gt0);
                for (int t = 1; t < ntiles && ok; ++t) {
                    score(gt0 + t);
                    if (ok) pv(gt0 + t - 1, t == 1);
                }
                if (ok) pv(gt0 + ntiles - 1, ntiles == 1);
                gt0 += ntiles;
                pos += ntiles;
                if constexpr (!RUNS) break;
            }
            if (!ok) *abort_flag = 1;
            tc_commit(drain);                  // nothing of this CTA's in tensor memory in flight
            mbar_wait(drain, 0);
        }
        __syncwarp();
    } else if ((warp & 3) < quarters) {
        // ---- softmax: thread = query row r, keys 64g..64g+63 of each tile -----------------
        const int q4 = warp & 3, g = warp >> 2;
        const int r = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t scol = (uint32_t)g * 64u;               // this half's first column
        const float sl = a.scale * 1.4426950408889634f;
        bool okw = true;
        int gt0 = 0;
        for (int pos = lo; pos < hi;) {
            int bh, t0, ntiles, slot;
            segment(pos, bh, t0, ntiles, slot);
            int n = n0;
            if constexpr (RUNS) n = n_s[bh / a.H];
            const int k_lo = t0 * FA_KEYS, k_hi = min((t0 + ntiles) * FA_KEYS, n);
            if (pos > lo) {   // a later segment: restage this row group's Q rows
                stage_q(bh, r, g);
                __syncwarp();
                if (lane == 0) mbar_arrive(q_ready);
            }
            float m_run = -INFINITY, l = 0.f;
            // Failures (a wait that ran out) are made uniform: within a warp by vote, across
            // the row group's two warps by the barriers that also publish the tile maxima and
            // close the segment, so both leave together.
            for (int t = 0; t < ntiles; ++t) {
                const int gt = gt0 + t, bsel = gt & 1;
                bool ok = okw && __all_sync(0xffffffffu, mbar_wait(&s_full[bsel], (uint32_t)(gt >> 1) & 1u));
                uint32_t raw_s[4][16];
                // valid keys of this half of the tile (the prefix may end inside the last tile)
                const int nv = min(64, max(0, k_hi - (k_lo + t * FA_KEYS + g * 64)));
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (ok) {
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        tmem_ld16_issue(trow + (uint32_t)bsel * 128u + scol + (uint32_t)(c * 16), raw_s[c]);
                    tmem_wait_ld();
                    if (nv == 64) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int j = 0; j < 16; ++j) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(raw_s[c][j]));
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                if (c * 16 + j < nv) mx[j & 3] = fmaxf(mx[j & 3], __uint_as_float(raw_s[c][j]));
                    }
                }
                xmax[bsel][g][r] = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                if (!named_bar_and(1 + q4, 64, ok)) { okw = false; break; }   // the row group's two warps
                const float mt = fmaxf(xmax[bsel][0][r], xmax[bsel][1][r]);
                const float m_new = fmaxf(m_run, mt * sl);
                const bool move = m_new > m_run + FA_RESCALE_LOG2 || m_run == -INFINITY;
                if (t > 0 && __any_sync(0xffffffffu, move)) {
                    // rescale this warp's half of its rows of O once P.V of the previous tile is done
                    if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(gt - 1) & 1], (uint32_t)((gt - 1) >> 1) & 1u))) {
                        okw = false;
                        continue;
                    }
                    tc_fence_after();
                    const float f = move ? ex2_approx_ftz(m_run - m_new) : 1.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[16];
                        tmem_ld16_issue(trow + o_col + scol + (uint32_t)(c * 16), o);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
                        tmem_st16(trow + o_col + scol + (uint32_t)(c * 16), o);
                    }
                    tmem_wait_st();
                    if (move) l *= f;
                }
                if (move) m_run = m_new;
                // P for this half tile into buffer bsel, once P.V of tile gt-2 has read it
                if (gt >= 2 &&
                    !__all_sync(0xffffffffu, mbar_wait(&pv_done[bsel], (uint32_t)((gt - 2) >> 1) & 1u))) {
                    okw = false;
                    continue;
                }
                uint8_t* pbase = sP + (size_t)bsel * FA_TILE + (size_t)g * FA_HALF;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 8; ++c) {   // 8 chunks of 8 keys
                    float e[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int key = c * 8 + j;
                        const float x = ex2_approx_ftz(fmaf(__uint_as_float(raw_s[key >> 4][key & 15]), sl, -m_run));
                        e[j] = key < nv ? x : 0.f;
                        ls[j & 3] += e[j];
                    }
                    uint4 u;
                    u.x = pack_bf16x2(e[0], e[1]);
                    u.y = pack_bf16x2(e[2], e[3]);
                    u.z = pack_bf16x2(e[4], e[5]);
                    u.w = pack_bf16x2(e[6], e[7]);
                    *reinterpret_cast<uint4*>(pbase + fa_sw128(r, c)) = u;
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[bsel]);
            }
            // ---- segment epilogue: the last P.V, then o (this half), m, l of each query row --
            bool bad = !okw;
            if (okw) {
                const int gl = gt0 + ntiles - 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[gl & 1], (uint32_t)(gl >> 1) & 1u))) bad = true;
            }
            tc_fence_after();
            bad = bad || *abort_flag;
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.flags, (uint32_t)EVS_FLAG_TIMEOUT);
            float* prow = a.part + (((size_t)bh * a.splits + slot) * a.q_stride + r) * (FA_DH + 2);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[16];
                tmem_ld16_issue(trow + o_col + scol + (uint32_t)(c * 16), o);
                tmem_wait_ld();
                if (r < a.Q && !bad) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2)   // rows are 8-byte aligned (130 floats apart)
                        *reinterpret_cast<float2*>(prow + g * 64 + c * 16 + j) =
                            make_float2(__uint_as_float(o[j]), __uint_as_float(o[j + 1]));
                }
            }
            if (g == 1) xsum[r] = l;
            const bool both_ok = named_bar_and(1 + q4, 64, !bad);
            if (g == 0 && r < a.Q) {
                prow[FA_DH] = bad ? -INFINITY : m_run * 0.6931471805599453f;   // natural units
                prow[FA_DH + 1] = bad ? 0.f : l + xsum[r];
            }
            tc_fence_before();   // this segment's TMEM reads precede the next segment's MMAs
            if (!both_ok) break;
            gt0 += ntiles;
            pos += ntiles;
            if constexpr (!RUNS) break;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        if (*abort_flag && lane == 0) {
            // an aborted pipeline may still have loads in flight into this CTA's ring: wait
            // (bounded) for the transactions of the last steps issued before the CTA exits
            for (int j = issued > a.stages ? issued - a.stages : 0; j < issued; ++j)
                mbar_wait(&full[j % a.stages], (uint32_t)(j / a.stages) & 1u);
        }
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- host side ------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 kv_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_kv_map(CUtensorMap* m, const void* base, int t_max, int bh) {
    auto fn = kv_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)FA_DH, (cuuint64_t)t_max, (cuuint64_t)bh};
    const cuuint64_t strides[2] = {(cuuint64_t)FA_DH * 2, (cuuint64_t)t_max * FA_DH * 2};
    const cuuint32_t box[3] = {64, FA_KEYS, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plan of a pass with Q (1..128) queries per sequence. Chunks first: the number of splits per
// (sequence, head) that minimises waves of one CTA per SM x (tiles per CTA + 2), a CTA's
// start-up and drain costing about two tiles' streaming. A persistent grid of FA_GRID CTAs
// over runs of tiles (each start-up paid once per SM, about one Q restage per run) is taken
// instead when its cost, tiles per SM + 3, is lower, or when the chunks take five or more
// waves; each (sequence, head) then meets at most FA_GRID / H + 2 runs.
AttnPlan attn_plan(int Q, int B, int H, int t_max, int smem_max) {
    AttnPlan p{};
    if (Q < 1 || Q > FA_ROWS || B > FA_MAX_B) return p;
    const int fixed = 1024 + 3 * FA_TILE + 16 * 8;   // align, Q, two P buffers, barriers (<= 16)
    int stages = (smem_max - fixed) / FA_TILE;
    if (stages > 3) stages = 3;
    if (stages < 2) return p;
    const long long total_tiles = (t_max + FA_KEYS - 1) / FA_KEYS;
    const long long bh = (long long)B * H;
    long long best = 1, best_cost = -1, best_waves = 1;
    for (long long s = 1; s <= total_tiles && s <= 4096; ++s) {
        const long long waves = (bh * s + FA_GRID - 1) / FA_GRID;
        const long long cost = waves * ((total_tiles + s - 1) / s + 2);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; best_waves = waves; }
    }
    p.n_q = FA_ROWS;
    // the persistent grid: every SM streams an equal run of the key tiles of all (sequence,
    // head) prefixes laid end to end; about one prefix boundary per run costs a Q restage
    const long long runs_cost = (bh * total_tiles + FA_GRID - 1) / FA_GRID + 3;
    if (best_waves >= 5 || runs_cost < best_cost) {
        p.runs = 1;
        p.splits = FA_GRID / H + 2;
    } else {
        p.runs = 0;
        p.splits = (int)best;
    }
    p.tiles = (int)((total_tiles + best - 1) / best);
    p.stages = stages;
    p.ncols = 512;
    p.smem = fixed + stages * FA_TILE;
    p.ok = 1;
    return p;
}

int attn_init() {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, attn_fa_kernel<true>) != cudaSuccess)
        return -1;
    const int dyn = optin - (int)fa.sharedSizeBytes;   // the larger static footprint of the two
    if (cudaFuncSetAttribute(attn_fa_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_fa_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
        return -1;
    return dyn;
}

bool launch_attn_tensor(evs_handle* h, int li, const Pass& p, const AttnPlan& plan) {
    const LayerDesc& L = h->layer[li];
    const int H = L.param;
    CUtensorMap tk, tv;
    if (!make_kv_map(&tk, L.kc, h->cfg.t_max, p.B * H) || !make_kv_map(&tv, L.vc, h->cfg.t_max, p.B * H))
        return false;
    FaArgs a{h->y, 3 * h->cfg.d, p.B, H, p.C * p.T, plan.splits, h->g.q_max, plan.stages,
             1.0f / sqrtf((float)FA_DH), h->kv_base, h->attn_part, h->flags};
    if (plan.runs)
        return launch_k(h, attn_fa_kernel<true>, dim3(FA_GRID), dim3(FA_THREADS), (size_t)plan.smem, tk, tv, a) ==
               cudaSuccess;
    return launch_k(h, attn_fa_kernel<false>, dim3(plan.splits, p.B * H), dim3(FA_THREADS), (size_t)plan.smem, tk,
                    tv, a) == cudaSuccess;
}

}  // namespace evs
