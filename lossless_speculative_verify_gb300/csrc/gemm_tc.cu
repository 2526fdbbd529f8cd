// Weight-streaming skinny projection on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA. Y[m][n] (+)= sum_k X[m][k] W[n][k] with X the block's activations (M =
// sequences x candidates x (gamma+1) rows, a few to a few hundred) and W an out-major
// weight matrix streamed from HBM exactly once per launch.
//
// Swap-AB: the weight tile is the 128-row A operand and the tokens are the N dimension of
// the MMA (16..256 per instruction, up to 512 in two accumulators), so the accumulator
// D[n][m] sits in TMEM with one output channel per lane. One CTA owns a 128-channel tile
// and a range of K; ranges of K are split across CTAs until the grid fills the 152 SMs.
// The splits of a tile form a thread-block cluster: each stores its fp32 partial tile to an
// L2-resident scratch, and after one cluster barrier each adds a run of token rows over the
// splits in a fixed order (deterministic). The in-projection of a FIR / IIR layer instead
// pushes channel slices through distributed shared memory and runs the mixer in the
// epilogue. Without a cluster, the last CTA to finish a tile adds the partial sums.
//
// Roles in a CTA of 128 threads: thread 0 issues TMA loads into a ring of stages, thread
// 32 issues the MMAs and releases stages with tcgen05.commit, then all four warps read
// their 32 TMEM lanes for the epilogue.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "evs_common.cuh"
#include "sm100_ptx.cuh"

namespace evs {

constexpr int TC_BM = 128;                    // output channels per tile (MMA M)
constexpr int TC_BK = 64;                     // K per stage: one 128-byte swizzled row of bf16
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2; // 16 KiB
#ifndef EVS_TC_SMEM_KB
#define EVS_TC_SMEM_KB 100     // shared-memory ring budget per CTA (two CTAs per SM)
#endif
#ifndef EVS_TC_CTA_TARGET
#define EVS_TC_CTA_TARGET 304  // CTAs one projection aims to fill (two per SM)
#endif
#ifndef EVS_TC_WIDE_NARROW
#define EVS_TC_WIDE_NARROW 0  // narrow outputs split beyond one cluster on the global path
#endif
#ifndef EVS_TC_MAX_SPLITS
#define EVS_TC_MAX_SPLITS 8
#endif
#ifndef EVS_TC_MIN_KB
#define EVS_TC_MIN_KB 2        // fewest 64-wide k-blocks a split may stream
#endif
constexpr int TC_SMEM_BUDGET = EVS_TC_SMEM_KB * 1024;
constexpr int TC_EXCLUSIVE_SMEM = 200 * 1024;   // dynamic shared memory of a CTA that needs its SM alone
#ifndef EVS_TC_KBS
#define EVS_TC_KBS 4          // 64-wide k-blocks per pipeline stage (longer contiguous row reads)
#endif
#ifndef EVS_TC_PACKED
#define EVS_TC_PACKED 0       // weights stored as contiguous [tile][k-block][128][64] blocks
#endif
#ifndef EVS_TC_ROTATE
#define EVS_TC_ROTATE 0       // start each tile's k loop at a different offset
#endif

struct TcArgs {
    float* Y;
    int ldy, M, N, kblocks, splits, n_pad, stages, accumulate, ncols, kbs;
    int cluster;      // 1: the splits of a tile form a cluster: partial tiles exchanged through
                      // the scratch (part) and reduced by row runs after a cluster barrier
    float* part;      // [splits][M][N] partial sums when splits > 1
    int* counters;    // [N / 128] arrival counters, zero between launches
    uint32_t* flags;
    // fused RMS norm: rows of the product scaled by 1/rms(h) from the producer's per-tile
    // sums of squares; the final writer of h leaves bf16(h) and its own sums of squares
    const float* ssq_in;   // [ssq_tiles][ssq_ld] or null
    int ssq_tiles, ssq_ld, norm_d;
    __nv_bfloat16* hb_out; // [M][hb_ld] or null
    int hb_ld;
    float* ssq_out;        // [N / 128][ssq_ld] or null
    // fused mixer of a FIR / IIR layer's in-projection (0 none, 1 FIR, 2 IIR): the product
    // v (or u) never reaches global memory; the mixer output goes to mix_out in bf16
    int mix, mix_C, mix_T, mix_commit, mix_param, d;   // param: FIR taps L or IIR poles N
    __nv_bfloat16* mix_out;                            // [M][d]
    const float* taps;
    float* tail;
    float* stage;
    const float2* lam;
    const float2* bq;
    const float2* cq;
    float2* state;
    float* uin;       // IIR, verify: the scan inputs u_t [M][d] kept for slicing
    // fused K/V write of an attention layer's QKV projection: columns [d, 3d) go to the
    // cache (one candidate) or the per-candidate side buffer instead of Y
    int kv, kv_H, kv_dh, kv_in_cache, kv_tmax, kv_C, kv_T;
    const int32_t* kv_base;
    __nv_bfloat16* kc;
    __nv_bfloat16* vc;
    __nv_bfloat16* ks;
    __nv_bfloat16* vs;
};

// The epilogue a launch runs, fixed at compile time: each instantiation carries only its own
// epilogue code, which runs once per CTA from a cold instruction cache (instruction-fetch
// stalls were a fifth of the stall cycles of the single kernel with every epilogue).
enum TcEpi : int {
    TC_EPI_PLAIN = 0,     // no split-K: TMEM straight to the outputs
    TC_EPI_CLUSTER = 1,   // split-K reduced by row runs within the cluster
    TC_EPI_GLOBAL = 2,    // split-K reduced by the last CTA of a tile
    TC_EPI_FIR = 3,       // in-projection with the FIR mixer
    TC_EPI_IIR = 4,       // in-projection with the modal IIR mixer
};

// KV: the launch writes K / V columns to the cache or side buffer (an attention layer's QKV).
// FL: the FIR mixer's filter length when fixed at compile time (0: up to 16, from the
// arguments), so that its once-per-CTA code holds only the taps it has.
template <int EPI, bool KV, int FL = 0>
__global__ void __launch_bounds__(128, 2)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot[1];
    __shared__ volatile int abort_flag[1];
    __shared__ int last_flag[1];
    __shared__ float rinv_s[512];
    __shared__ __align__(16) float red_s[4 * 512];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int b_bytes = p.n_pad * 128;
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)p.stages * p.kbs * TC_A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)p.stages * p.kbs * b_bytes);
    uint64_t* empty = full + p.stages;
    uint64_t* done = empty + p.stages;

    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int n0 = tile * TC_BM;
    const int kb0 = (int)((long long)p.kblocks * split / p.splits);
    const int kb1 = (int)((long long)p.kblocks * (split + 1) / p.splits);
    const int nkb = kb1 - kb0;
    const int nst = (nkb + p.kbs - 1) / p.kbs;              // pipeline steps of up to kbs k-blocks
    const int rot = EVS_TC_ROTATE ? (tile * 5) % nst : 0;    // spread concurrent row offsets
    const int a_stage = TC_A_BYTES * p.kbs, b_stage = b_bytes * p.kbs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, (uint32_t)p.ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 0) {
        // ---- producer: TMA ring ------------------------------------------------------
        const uint64_t pol_w = policy_evict_first();   // weights: read once
        const uint64_t pol_x = policy_evict_last();    // activations: read by every tile
        auto load = [&](int i, bool a, bool b) {
            const int s = i % p.stages;
            const int st = (i + rot) % nst;
            const int k0 = kb0 + st * p.kbs;
            const int cnt = min(p.kbs, kb1 - k0);
            if (a) mbar_arrive_expect_tx(&full[s], (uint32_t)(cnt * (TC_A_BYTES + b_bytes)));
            for (int j = 0; j < cnt; ++j) {
                const int k = (k0 + j) * TC_BK;
                if (a) {
#if EVS_TC_PACKED
                    tma_load_2d(sA + (size_t)s * a_stage + (size_t)j * TC_A_BYTES, &tmA, 0,
                                (tile * p.kblocks + k0 + j) * TC_BM, &full[s], pol_w);
#else
                    tma_load_2d(sA + (size_t)s * a_stage + (size_t)j * TC_A_BYTES, &tmA, k, n0, &full[s], pol_w);
#endif
                }
                if (b)
                    for (int r = 0; r < p.n_pad; r += 256)
                        tma_load_2d(sB + (size_t)s * b_stage + (size_t)j * b_bytes + (size_t)r * 128, &tmB, k, r,
                                    &full[s], pol_x);
            }
        };
        // weights do not depend on the previous kernel: fill the ring with them before
        // waiting for it, then add the activations
        const int pre = min(p.stages, nst);
        for (int i = 0; i < pre; ++i) load(i, true, false);
        pdl_wait();
        for (int i = 0; i < pre; ++i) load(i, false, true);
        for (int i = pre; i < nst; ++i) {
            const int s = i % p.stages;
            const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
            if (!mbar_wait(&empty[s], ph ^ 1u)) { *abort_flag = 1; break; }
            load(i, true, true);
        }
    } else if (threadIdx.x == 32) {
        // ---- MMA issuer ------------------------------------------------------------------
        const int n_hi = p.n_pad > 256 ? p.n_pad - 256 : 0;
        const int n_lo = p.n_pad - n_hi;
        const uint32_t id_lo = idesc_bf16_f32(TC_BM, n_lo);
        const uint32_t id_hi = idesc_bf16_f32(TC_BM, n_hi > 0 ? n_hi : 16);
        for (int i = 0; i < nst; ++i) {
            const int s = i % p.stages;
            const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
            if (!mbar_wait(&full[s], ph)) { *abort_flag = 1; break; }
            tc_fence_after();
            const int st = (i + rot) % nst;
            const int cnt = min(p.kbs, kb1 - (kb0 + st * p.kbs));
            for (int j = 0; j < cnt; ++j) {
                const uint32_t a0 = smem_u32(sA + (size_t)s * a_stage + (size_t)j * TC_A_BYTES);
                const uint32_t b0 = smem_u32(sB + (size_t)s * b_stage + (size_t)j * b_bytes);
#pragma unroll
                for (int kk = 0; kk < TC_BK / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(a0 + kk * 32);
                    const uint32_t acc = (i > 0 || j > 0 || kk > 0) ? 1u : 0u;
                    tc_mma_f16(tmem, ad, smem_desc_sw128(b0 + kk * 32), id_lo, acc);
                    if (n_hi > 0)
                        tc_mma_f16(tmem + 256, ad, smem_desc_sw128(b0 + 256 * 128 + kk * 32), id_hi, acc);
                }
            }
            tc_commit(&empty[s]);
        }
        tc_commit(done);
    }

    // ---- epilogue: lane = output channel, columns = tokens ---------------------------------
    pdl_wait();
    // Mixer of a FIR / IIR in-projection: this CTA's channel slice [mc_lo, mc_lo + mcw) (the
    // whole tile without split-K). The parameters and carried state of each thread's first
    // items are loaded here, while the mainloop still runs.
    const int mc_lo = (int)(128LL * split / p.splits);
    const int mcw = (int)(128LL * (split + 1) / p.splits) - mc_lo;
    const int mT = p.mix_T > 0 ? p.mix_T : 1, mgroups = p.M / mT;
    // FIR item: one (group g, block position t, channel c), channels fastest: its taps w[j],
    // zero past the filter length
    constexpr int KL = FL > 0 ? FL : 16;   // FIR taps held per item
    auto fir_load = [&](int item, float (&w)[KL]) {
        const int L = FL > 0 ? FL : p.mix_param;
        const bool on = item < mgroups * mT * mcw;
        const int n = n0 + mc_lo + (on ? item % mcw : 0);
#pragma unroll
        for (int j = 0; j < KL; ++j) w[j] = (on && j < L) ? p.taps[(size_t)n * L + j] : 0.f;
    };
    // IIR item: one (g, channel, quad of four poles); pole lambda, input weight B, readout
    // weight C and carried state of the quad's poles
    auto iir_load = [&](int it, float2 (&l)[4], float2 (&bq)[4], float2 (&cq)[4], float2 (&sv)[4]) {
        const int N = p.mix_param, Q = N / 4;
        const bool on = it < mgroups * mcw * Q;
        const int k0 = on ? (it % Q) * 4 : 0, n = n0 + mc_lo + (on ? (it / Q) % mcw : 0);
        const int b = on ? (it / (Q * mcw)) / p.mix_C : 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            l[k] = on ? p.lam[(size_t)n * N + k0 + k] : make_float2(0.f, 0.f);
            bq[k] = on ? p.bq[(size_t)n * N + k0 + k] : make_float2(0.f, 0.f);
            cq[k] = on ? p.cq[(size_t)n * N + k0 + k] : make_float2(0.f, 0.f);
            sv[k] = on ? p.state[((size_t)b * p.d + n) * N + k0 + k] : make_float2(0.f, 0.f);
        }
    };
    float fw[KL];
    float2 il[4], ib[4], ic[4], is[4];
    if constexpr (EPI == TC_EPI_FIR) {
        fir_load(threadIdx.x, fw);
    } else if constexpr (EPI == TC_EPI_IIR) {
        iir_load(threadIdx.x, il, ib, ic, is);
    }
    if (p.ssq_in && warp >= 2) {
        // 1/rms of each token row from the per-tile sums of squares of h, computed by the two
        // warps that are idle during the mainloop: one row per lane (the loads of a tile are
        // coalesced across the lanes), up to 32 tiles' loads in flight before any is summed
        for (int m0 = (warp - 2) * 32; m0 < p.M; m0 += 64) {
            const int m = m0 + lane;
            if (m < p.M) {
                float ss = 0.f;
                for (int t0 = 0; t0 < p.ssq_tiles; t0 += 32) {
                    float v[32];
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        v[u] = t0 + u < p.ssq_tiles ? p.ssq_in[(size_t)(t0 + u) * p.ssq_ld + m] : 0.f;
#pragma unroll
                    for (int u = 0; u < 32; ++u) ss += v[u];
                }
                rinv_s[m] = rsqrtf(ss / (float)p.norm_d + 1e-6f);
            }
        }
    }
    __syncwarp();
    const bool ok = mbar_wait(done, 0);
    tc_fence_after();
    const bool bad = !ok || *abort_flag;
    if (bad && threadIdx.x == 0) atomicOr(p.flags, (uint32_t)EVS_FLAG_TIMEOUT);
    __syncthreads();
    // Rows of the fused K/V write: the destination offset of each token row (the channel's
    // share added per thread), -1 past the end of the cache. Shares red_s with the sums of
    // squares, which a K/V-writing launch never produces.
    long long* kv_row = reinterpret_cast<long long*>(red_s);
    const bool kv_ch = KV && n0 + (int)threadIdx.x >= p.d;   // this thread's channel is K or V
    long long kv_col = 0;
    __nv_bfloat16* kv_dst = nullptr;
    if constexpr (KV) {
        for (int m = threadIdx.x; m < p.M; m += blockDim.x) {
            const int bc = m / p.kv_T, i = m % p.kv_T, b = bc / p.kv_C;
            long long o;
            if (p.kv_in_cache) {
                const int t = p.kv_base[b] + i;
                o = t < p.kv_tmax ? ((long long)b * p.kv_H * p.kv_tmax + t) * p.kv_dh : -1;
            } else {
                o = ((long long)bc * p.kv_H * p.kv_T + i) * p.kv_dh;
            }
            kv_row[m] = o;
        }
        if (kv_ch) {
            const int c2 = n0 + (int)threadIdx.x - p.d, which = c2 / p.d, col = c2 % p.d;
            const int hh = col / p.kv_dh, e = col % p.kv_dh;
            kv_col = (long long)hh * (p.kv_in_cache ? p.kv_tmax : p.kv_T) * p.kv_dh + e;
            kv_dst = p.kv_in_cache ? (which ? p.vc : p.kc) : (which ? p.vs : p.ks);
        }
        __syncthreads();
    }
    // The residual a row adds (0 without accumulation); callers load a batch of rows' values
    // before finishing any of them.
    auto resid = [&](int m, int nl) -> float {
        return (p.accumulate && m < p.M) ? p.Y[(size_t)m * p.ldy + n0 + nl] : 0.f;
    };
    // One output value: row scale, store (plus the residual res), bf16 copy, and this warp's
    // share of the row's sum of squares. All lanes of a warp call it for the same m with
    // consecutive channels; nl is the calling thread's index.
    auto finish = [&](int m, int nl, float v, float res, bool live) {
        if (p.ssq_in) v *= rinv_s[m];
        float out = v;
        if (kv_ch) {
            if (live) {
                const long long r = kv_row[m];
                if (r >= 0)
                    kv_dst[r + kv_col] = __float2bfloat16_rn(out);
                else
                    atomicOr(p.flags, (uint32_t)EVS_FLAG_KV_OVERFLOW);
            }
            return;
        }
        if (live) {
            out += res;
            p.Y[(size_t)m * p.ldy + n0 + nl] = out;
            if (p.hb_out) p.hb_out[(size_t)m * p.hb_ld + n0 + nl] = __float2bfloat16_rn(out);
        }
        if (p.ssq_out) {
            const float sq = warp_sum(live ? out * out : 0.f);
            if ((nl & 31) == 0) red_s[(nl >> 5) * 512 + m] = sq;
        }
    };
    // Four consecutive channels 4*lane.. of one row (a warp covers the 128-channel row):
    // float4 residual and stores, the row's sum of squares reduced within the warp.
    const long long kv_col4 = [&]() -> long long {
        if (!kv_ch) return 0;
        const int c2 = n0 + 4 * lane - p.d, col = c2 % p.d;
        return (long long)(col / p.kv_dh) * (p.kv_in_cache ? p.kv_tmax : p.kv_T) * p.kv_dh + col % p.kv_dh;
    }();
    auto resid4 = [&](int m) -> float4 {
        return p.accumulate ? *reinterpret_cast<const float4*>(p.Y + (size_t)m * p.ldy + n0 + 4 * lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto finish4 = [&](int m, float4 v, float4 res, bool live) {
        if (p.ssq_in) {
            const float r = rinv_s[m];
            v.x *= r; v.y *= r; v.z *= r; v.w *= r;
        }
        if (kv_ch) {
            if (live) {
                const long long r = kv_row[m];
                if (r >= 0) {
                    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
                    uint2 u;
                    u.x = *reinterpret_cast<const uint32_t*>(&a);
                    u.y = *reinterpret_cast<const uint32_t*>(&b);
                    *reinterpret_cast<uint2*>(kv_dst + r + kv_col4) = u;
                } else if (lane == 0) {
                    atomicOr(p.flags, (uint32_t)EVS_FLAG_KV_OVERFLOW);
                }
            }
            return;
        }
        float4 out = make_float4(v.x + res.x, v.y + res.y, v.z + res.z, v.w + res.w);
        if (live) {
            *reinterpret_cast<float4*>(p.Y + (size_t)m * p.ldy + n0 + 4 * lane) = out;
            if (p.hb_out) {
                const __nv_bfloat162 a = __floats2bfloat162_rn(out.x, out.y),
                                     b = __floats2bfloat162_rn(out.z, out.w);
                uint2 u;
                u.x = *reinterpret_cast<const uint32_t*>(&a);
                u.y = *reinterpret_cast<const uint32_t*>(&b);
                *reinterpret_cast<uint2*>(p.hb_out + (size_t)m * p.hb_ld + n0 + 4 * lane) = u;
            }
        }
        if (p.ssq_out) {
            const float sq = warp_sum(live ? out.x * out.x + out.y * out.y + out.z * out.z + out.w * out.w : 0.f);
            if (lane == 0) p.ssq_out[(size_t)tile * p.ssq_ld + m] = sq;
        }
    };
    int own_lo = 0, own_hi = 0;   // token rows whose sums of squares this CTA completes
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int nl_lane = warp * 32 + lane;
    if constexpr (EPI == TC_EPI_FIR || EPI == TC_EPI_IIR) {
        // ---- in-projection + mixer: gather this CTA's channel slice of v for every token
        // row (whole tile without split-K; a 1/S share of the channels with a cluster), then
        // one thread per (sequence-candidate, channel) runs the FIR / modal IIR over time
        float* park = reinterpret_cast<float*>(smem);
        const int S = p.splits;
        const int c_lo = (int)(128LL * split / S), c_hi = (int)(128LL * (split + 1) / S);
        const int cw = c_hi - c_lo;
        const int cwm = (TC_BM + S - 1) / S;                         // slot row stride
        // S == 1: park = [M][128] the whole tile; else park = [S][M][cwm] the partials of
        // this CTA's channel slice as pushed by every rank, then vals = [M][cw] their sum
        float* vals = S == 1 ? park : park + (size_t)S * p.M * cwm;
        if (S == 1) {
            for (int c0 = 0; c0 < p.M; c0 += 16) {
                float v[16];
                tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < p.M) park[(size_t)(c0 + j) * TC_BM + nl_lane] = v[j];
            }
        } else {
            const int own = ((nl_lane + 1) * S - 1) / TC_BM;         // rank owning this channel
            const int own_lo = (int)(128LL * own / S);
            const uint32_t dst = map_peer(smem_u32(park), (uint32_t)own) +
                                 (uint32_t)((size_t)split * p.M * cwm + nl_lane - own_lo) * 4u;
            cluster_sync();                       // every rank's mainloop is done: rings free
            for (int c0 = 0; c0 < p.M; c0 += 16) {
                float v[16];
                tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < p.M) st_peer_f32(dst + (uint32_t)((c0 + j) * cwm) * 4u, v[j]);
            }
            cluster_sync();                       // every push has landed
            for (int idx = threadIdx.x; idx < p.M * cw; idx += blockDim.x) {
                const int m = idx / cw, c = idx % cw;
                float acc = 0.f;
                for (int sp = 0; sp < S; ++sp) acc += park[((size_t)sp * p.M + m) * cwm + c];
                vals[idx] = acc;
            }
        }
        __syncthreads();
        const int vld = S == 1 ? TC_BM : cw;      // row stride of vals
        const int T = p.mix_T, groups = p.M / T;
        const int voff = S == 1 ? c_lo : 0;       // column of this CTA's first channel in vals
        // the mixer's input x_t of block row (g, t), channel column c of vals (1/rms applied)
        auto xin = [&](int g, int t, int c) -> float {
            return vals[(size_t)(g * T + t) * vld + voff + c] * (p.ssq_in ? rinv_s[g * T + t] : 1.f);
        };
        if constexpr (EPI == TC_EPI_FIR) {
            // FIR, y_t = sum_j w_j x_{t-j}: no recurrence, so one thread per (group, block
            // position, channel), channels fastest (coalesced stores); x_{-m} for m >= 1 is
            // row L-1-m of the carried tail
            const int L = FL > 0 ? FL : p.mix_param;
            const int items = groups * T * cw;
            for (int it = threadIdx.x; it < items && !bad; it += blockDim.x) {
                if (it != (int)threadIdx.x && blockDim.x % cw != 0) fir_load(it, fw);   // else same channel
                const int c = it % cw, t = (it / cw) % T, g = it / (cw * T);
                const int n = n0 + c_lo + c, b = g / p.mix_C;
                const float* tl = p.tail + (size_t)b * (L - 1) * p.d + n;
                float xv[KL];   // x_{t-j}: every input's load issued before the sum
#pragma unroll
                for (int j = 0; j < KL; ++j)
                    xv[j] = j >= L ? 0.f : (t - j >= 0 ? xin(g, t - j, c) : tl[(size_t)(L - 1 - j + t) * p.d]);
                float y = fw[0] * xv[0];
#pragma unroll
                for (int j = 1; j < KL; ++j)
                    if (j < L) y = fmaf(fw[j], xv[j], y);
                p.mix_out[((size_t)g * T + t) * p.d + n] = __float2bfloat16_rn(y);
                if (!p.mix_commit) {   // stage rows [tail || block inputs] of this group
                    float* st = p.stage + (size_t)g * (L - 1 + T) * p.d + n;
                    st[(size_t)(L - 1 + t) * p.d] = xv[0];
                    if (t == 0) {   // every row's load issued before any store
                        float tv[KL];
#pragma unroll
                        for (int r = 0; r < KL - 1; ++r) tv[r] = r < L - 1 ? tl[(size_t)r * p.d] : 0.f;
#pragma unroll
                        for (int r = 0; r < KL - 1; ++r)
                            if (r < L - 1) st[(size_t)r * p.d] = tv[r];
                    }
                }
            }
            if (p.mix_commit && L > 1) {
                // new tail rows i = x_{T-(L-1)+i} (row i+T of the old tail while that is
                // negative). Items (sequence, row, channel) in rounds; a round reads all its
                // values before writing any, and the old rows it reads are written only by
                // the same or a later round (rows ascend with the item index).
                const int tail_items = (groups / p.mix_C) * (L - 1) * cw;   // one per sequence
                for (int r0 = 0; r0 < tail_items; r0 += 4 * (int)blockDim.x) {
                    float nv[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int it = r0 + threadIdx.x + u * blockDim.x;
                        nv[u] = 0.f;
                        if (it < tail_items) {
                            const int c = it % cw, i = (it / cw) % (L - 1), bq = it / (cw * (L - 1));
                            const int g = bq * p.mix_C, t = T - (L - 1) + i, n = n0 + c_lo + c;
                            nv[u] = t >= 0 ? xin(g, t, c) : p.tail[((size_t)bq * (L - 1) + (i + T)) * p.d + n];
                        }
                    }
                    __syncthreads();
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int it = r0 + threadIdx.x + u * blockDim.x;
                        if (it < tail_items && !bad) {
                            const int c = it % cw, i = (it / cw) % (L - 1), bq = it / (cw * (L - 1));
                            p.tail[((size_t)bq * (L - 1) + i) * p.d + n0 + c_lo + c] = nv[u];
                        }
                    }
                    __syncthreads();
                }
            }
        } else {
            // modal IIR: a thread per (group, channel, quad of four poles); the readout of
            // eight positions at a time is reduced over the channel's N/4 lanes side by side.
            // A verify pass keeps the inputs u_t (slicing recomputes s_k from them).
            const int N = p.mix_param, Q = N / 4;
            const int items = groups * cw * Q;
            const int span = (items + 31) / 32 * 32;              // whole warps take part
            for (int it = threadIdx.x; it < span; it += blockDim.x) {
                if (it != (int)threadIdx.x) iir_load(it, il, ib, ic, is);
                const bool on = it < items && !bad;
                const int k0 = (it % Q) * 4, c = (it / Q) % cw, g = min(it / (Q * cw), groups - 1);
                const int n = n0 + c_lo + c;
                const float* vr = vals + (size_t)g * T * vld + voff + c;
                const float* rr = rinv_s + g * T;
                for (int t0 = 0; t0 < T; t0 += 8) {
                    float q[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float y = 0.f;
                        if (t0 + u < T) {
                            const float uu = on ? vr[(size_t)(t0 + u) * vld] * (p.ssq_in ? rr[t0 + u] : 1.f) : 0.f;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                is[k] = make_float2(fmaf(il[k].x, is[k].x, fmaf(-il[k].y, is[k].y, ib[k].x * uu)),
                                                    fmaf(il[k].x, is[k].y, fmaf(il[k].y, is[k].x, ib[k].y * uu)));
                                y = fmaf(ic[k].x, is[k].x, fmaf(-ic[k].y, is[k].y, y));
                            }
                            if (on && !p.mix_commit && k0 == 0) p.uin[((size_t)g * T + t0 + u) * p.d + n] = uu;
                        }
                        q[u] = y;
                    }
                    for (int o = Q >> 1; o > 0; o >>= 1)
#pragma unroll
                        for (int u = 0; u < 8; ++u) q[u] += __shfl_xor_sync(0xffffffffu, q[u], o);
                    if (on && k0 == 0) {
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            if (t0 + u < T) p.mix_out[((size_t)g * T + t0 + u) * p.d + n] = __float2bfloat16_rn(q[u]);
                    }
                }
                if (on && p.mix_commit) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) p.state[((size_t)(g / p.mix_C) * p.d + n) * N + k0 + k] = is[k];
                }
            }
        }
    } else if constexpr (EPI == TC_EPI_PLAIN) {
        for (int c0 = 0; c0 < p.M; c0 += 16) {
            float v[16], r[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = resid(c0 + j, nl_lane);
            tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < p.M) finish(c0 + j, nl_lane, v[j], r[j], !bad);
        }
        own_hi = p.M;
    } else if constexpr (EPI == TC_EPI_CLUSTER) {
        // split-K within the cluster through L2: every rank stores its partial tile to the
        // scratch, one cluster barrier, then each rank adds a run of rows over the ranks in
        // rank order (deterministic) and finishes them: a row per warp, four channels a lane
        const int S = p.splits;
        float* mine = p.part + ((size_t)tile * S + split) * p.M * TC_BM;
        for (int c0 = 0; c0 < p.M; c0 += 16) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < p.M) mine[(size_t)(c0 + j) * TC_BM + nl_lane] = v[j];
        }
        cluster_sync();                           // every rank's partial tile is in L2
        const int per = (p.M + S - 1) / S;
        const int lo = split * per, hi = min(p.M, lo + per);
        const float* base = p.part + (size_t)tile * S * p.M * TC_BM;
        for (int m = lo + warp; m < hi; m += 4) {
            const float4 res = resid4(m);
            float4 x[8];
#pragma unroll
            for (int sp = 0; sp < 8; ++sp)
                x[sp] = sp < S ? __ldcg(reinterpret_cast<const float4*>(base + ((size_t)sp * p.M + m) * TC_BM) + lane)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            float4 acc = x[0];
#pragma unroll
            for (int sp = 1; sp < 8; ++sp) {
                acc.x += x[sp].x;
                acc.y += x[sp].y;
                acc.z += x[sp].z;
                acc.w += x[sp].w;
            }
            finish4(m, acc, res, !bad);
        }
    } else {
        const int n = n0 + nl_lane;
        float* mine = p.part + (size_t)split * p.M * p.N;
        for (int c0 = 0; c0 < p.M; c0 += 16) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = c0 + j;
                if (m < p.M && !bad) mine[(size_t)m * p.N + n] = v[j];
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) *last_flag = (atomicAdd(&p.counters[tile], 1) == p.splits - 1);
        __syncthreads();
        if (*last_flag) {
            __threadfence();
            // four rows at a time, every split's value requested before any is summed
            for (int m0 = 0; m0 < p.M; m0 += 4) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f}, rv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) rv[u] = resid(m0 + u, nl_lane);
                for (int sp = 0; sp < p.splits; ++sp) {
                    float v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        v[u] = (m0 + u < p.M) ? __ldcg(p.part + ((size_t)sp * p.M + m0 + u) * p.N + n) : 0.f;
#pragma unroll
                    for (int u = 0; u < 4; ++u) acc[u] += v[u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (m0 + u < p.M) finish(m0 + u, nl_lane, acc[u], rv[u], !bad);
            }
            if (threadIdx.x == 0) p.counters[tile] = 0;
            own_hi = p.M;
        }
    }
    if (p.ssq_out && !(p.splits > 1 && p.cluster)) {
        __syncthreads();
        auto put = [&](int lo, int hi) {
            for (int m = lo + threadIdx.x; m < hi; m += blockDim.x)
                p.ssq_out[(size_t)tile * p.ssq_ld + m] =
                    red_s[m] + red_s[512 + m] + red_s[1024 + m] + red_s[1536 + m];
        };
        put(own_lo, own_hi);   // (the cluster path wrote its rows' sums directly)
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.ncols);
    }
}

// ---- host side ------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    }
    return fn;
}

// Row-major bf16 matrix [rows][cols] as a 2-D tensor map with a box of box_rows x 64 and
// 128-byte swizzle. Returns false if the driver rejects it.
static bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {TC_BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Opt the kernel into the largest dynamic shared memory the device allows next to its
// static shared memory; returns that size in bytes, or -1 on failure.
using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, TcArgs);
// [KV][epilogue]; the mixers never write K / V
static const TcKernel kTcKernels[2][5] = {
    {gemm_tc_kernel<TC_EPI_PLAIN, false>, gemm_tc_kernel<TC_EPI_CLUSTER, false>,
     gemm_tc_kernel<TC_EPI_GLOBAL, false>, gemm_tc_kernel<TC_EPI_FIR, false>, gemm_tc_kernel<TC_EPI_IIR, false>},
    {gemm_tc_kernel<TC_EPI_PLAIN, true>, gemm_tc_kernel<TC_EPI_CLUSTER, true>,
     gemm_tc_kernel<TC_EPI_GLOBAL, true>, nullptr, nullptr}};

// FIR mixers of the filter lengths the layers use, fixed at compile time
static const TcKernel kTcFir3 = gemm_tc_kernel<TC_EPI_FIR, false, 3>;
static const TcKernel kTcFir7 = gemm_tc_kernel<TC_EPI_FIR, false, 7>;

// The instantiation for a launch's arguments.
static TcKernel tc_kernel_for(const TcArgs& a) {
    if (a.mix == 1) return a.mix_param == 3 ? kTcFir3 : a.mix_param == 7 ? kTcFir7 : kTcKernels[0][TC_EPI_FIR];
    if (a.mix == 2) return kTcKernels[0][TC_EPI_IIR];
    const int e = a.splits == 1 ? TC_EPI_PLAIN : (a.cluster ? TC_EPI_CLUSTER : TC_EPI_GLOBAL);
    return kTcKernels[a.kv ? 1 : 0][e];
}

int gemm_tc_init() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return -1;
    TcKernel all[12];
    int n = 0;
    for (const auto& row : kTcKernels)
        for (TcKernel k : row)
            if (k) all[n++] = k;
    all[n++] = kTcFir3;
    all[n++] = kTcFir7;
    int dyn = optin;
    for (int i = 0; i < n; ++i) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, all[i]) != cudaSuccess) return -1;
        dyn = std::min(dyn, optin - (int)fa.sharedSizeBytes);
    }
    for (int i = 0; i < n; ++i)
        if (cudaFuncSetAttribute(all[i], cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess) return -1;
    return dyn;
}

// Split K only as far as each CTA still streams at least EVS_TC_MIN_KB k-blocks, and no
// further than about two CTAs per SM: past that the partial-sum round trip and the per-CTA
// start-up cost more than the extra parallelism returns.
int tc_cta_target() { return EVS_TC_CTA_TARGET; }

int tc_splits(int N, int K) {
    const int tiles = N / TC_BM, kblocks = K / TC_BK;
    int s = EVS_TC_CTA_TARGET / tiles;
    if (s > kblocks / EVS_TC_MIN_KB) s = kblocks / EVS_TC_MIN_KB;
    // stay within one portable cluster unless that leaves most SMs idle (narrow outputs such
    // as the LM head), where the global partial-sum path splits further
    if (s > EVS_TC_MAX_SPLITS && (tiles * EVS_TC_MAX_SPLITS >= 152 || !EVS_TC_WIDE_NARROW)) s = EVS_TC_MAX_SPLITS;
    if (s < 1) s = 1;
    return s;
}

// Launch shape of one projection: token padding, split-K, k-blocks per stage, ring depth,
// TMEM columns and dynamic shared memory.
struct TcShape {
    int n_pad, tiles, kblocks, splits, kbs, stages, ncols, cluster;
    size_t smem;
};

// Partial-sum floats a shape needs in global scratch (splits > 1 without the cluster path).
static size_t tc_part_floats(const TcShape& t, int M, int N) {
    return (t.splits > 1 && !t.cluster) ? (size_t)t.splits * M * N : 0;
}

static TcShape tc_shape(int M, int N, int K, size_t part_cap = (size_t)-1, int max_splits = 1 << 30,
                        bool allow_cluster = true) {
    TcShape t{};
    // tokens padded to the MMA's N granularity; above 256 two accumulators of 256 columns
    t.n_pad = M > 256 ? 512 : (M + 15) / 16 * 16;
    t.tiles = N / TC_BM;
    t.kblocks = K / TC_BK;
    t.splits = tc_splits(N, K);
    if (t.splits > max_splits) t.splits = max_splits;
    const int per = (t.kblocks + t.splits - 1) / t.splits;
    t.kbs = EVS_TC_KBS;
    const int kb_bytes = TC_A_BYTES + t.n_pad * 128;
    while (t.kbs > 1 && (t.kbs > per || 2 * t.kbs * kb_bytes > TC_SMEM_BUDGET)) t.kbs >>= 1;
    const int steps = (per + t.kbs - 1) / t.kbs;
    t.stages = TC_SMEM_BUDGET / (t.kbs * kb_bytes);
    if (t.stages > steps) t.stages = steps;
    if (t.stages < 1) t.stages = 1;
    t.ncols = 32;
    while (t.ncols < t.n_pad) t.ncols <<= 1;
    t.smem = (size_t)t.stages * t.kbs * kb_bytes + 1024 + (2 * t.stages + 1) * 8;
    // a 512-column accumulator takes all of an SM's tensor memory. Such a CTA gets the SM to
    // itself (more shared memory than leaves room for any other projection or attention
    // CTA): otherwise a CTA could hold the columns while it waits on a cluster peer or on its
    // predecessor kernel, with the CTA it waits for stuck in its own allocation.
    if (t.ncols > 256) t.smem = std::max(t.smem, (size_t)TC_EXCLUSIVE_SMEM);
    // cluster reduction when the splits fit a portable cluster and the scratch holds every
    // partial tile of the launch
    t.cluster = allow_cluster && t.splits > 1 && t.splits <= 8 && (size_t)N * t.splits * M <= part_cap;
    if (tc_part_floats(t, M, N) > part_cap && t.splits > 1) {
        // scratch too small for this many partial tiles: fewer splits
        int s = (int)(part_cap / ((size_t)M * N));
        return tc_shape(M, N, K, part_cap, s < 1 ? 1 : s, allow_cluster);
    }
    return t;
}

static bool launch_tc(const TcShape& t, const CUtensorMap& ta, const CUtensorMap& tb, const TcArgs& a,
                      cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(t.tiles, t.splits);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = t.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (t.cluster) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = (unsigned)t.splits;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, tc_kernel_for(a), ta, tb, a) == cudaSuccess;
}

bool gemm_tc_supported(int M, int N, int K) {
    return M >= 1 && M <= 512 && N % TC_BM == 0 && K % TC_BK == 0 && N > 0 && K > 0;
}

// Returns false (nothing launched) if a tensor map could not be built.
bool launch_gemm_tc(evs_handle* h, const void* X, int x_rows, const void* W, float* Y, int M, int N, int K,
                    int ldy, int accumulate, const GemmFuse* fz, int* fused) {
    if (fused) *fused = 0;
    // the cluster reduction finishes four channels per lane with 16-byte stores
    const bool vec_ok = ((uintptr_t)Y % 16 == 0) && ldy % 4 == 0 &&
                        (!fz || !fz->hb_out || ((uintptr_t)fz->hb_out % 8 == 0 && fz->hb_ld % 4 == 0));
    const TcShape t = tc_shape(M, N, K, h->gemm_part_floats, 1 << 30, vec_ok);
    CUtensorMap ta, tb;
#if EVS_TC_PACKED
    if (!make_map(&ta, W, (uint64_t)N * K / TC_BK, (uint64_t)TC_BK, TC_BM)) return false;
#else
    if (!make_map(&ta, W, (uint64_t)N, (uint64_t)K, TC_BM)) return false;
#endif
    if (!make_map(&tb, X, (uint64_t)x_rows, (uint64_t)K, (uint32_t)(t.n_pad < 256 ? t.n_pad : 256))) return false;
    if ((int)t.smem > h->tc_smem_max) return false;
    TcArgs a{};
    a.Y = Y; a.ldy = ldy; a.M = M; a.N = N; a.kblocks = t.kblocks; a.splits = t.splits; a.n_pad = t.n_pad;
    a.stages = t.stages; a.accumulate = accumulate; a.ncols = t.ncols; a.kbs = t.kbs; a.cluster = t.cluster;
    a.part = h->gemm_part; a.counters = h->gemm_counters; a.flags = h->flags;
    a.d = h->cfg.d;
    int did = 0;
    if (fz) {
        a.ssq_in = fz->ssq_in;
        a.ssq_tiles = fz->ssq_tiles;
        a.ssq_ld = fz->ssq_ld;
        a.norm_d = fz->norm_d;
        a.hb_out = fz->hb_out;
        a.hb_ld = fz->hb_ld;
        a.ssq_out = fz->ssq_out;
        const Pass* ps = fz->pass;
        const size_t ring = (size_t)t.stages * t.kbs * (TC_A_BYTES + t.n_pad * 128);
        if (fz->mix_layer >= 0 && ps) {
            // the mixer runs in the epilogue when the whole partial tile (plus the reduced
            // channel slice) sits in the ring at once and the split is a cluster or none
            const LayerDesc& L = h->layer[fz->mix_layer];
            const evs_layer_weights& LW = h->w.layer[fz->mix_layer];
            const int cw = (TC_BM + t.splits - 1) / t.splits;
            size_t need = t.splits > 1 ? (size_t)(t.splits + 1) * M * cw * 4 : (size_t)M * TC_BM * 4;

            const bool shape_ok = (t.splits == 1 || t.cluster) && need <= ring && M % ps->T == 0 &&
                                  (L.kind == EVS_LAYER_FIR || (L.param % 4 == 0 && L.param <= 32));
            if (shape_ok) {
                a.mix = L.kind == EVS_LAYER_FIR ? 1 : 2;
                a.mix_C = ps->C;
                a.mix_T = ps->T;
                a.mix_commit = ps->commit;
                a.mix_param = L.param;
                a.mix_out = (__nv_bfloat16*)h->act;
                a.taps = LW.fir_taps;
                a.tail = L.tail;
                a.stage = L.stage;
                a.lam = (const float2*)LW.iir_lambda;
                a.bq = (const float2*)LW.iir_b;
                a.cq = (const float2*)LW.iir_c;
                a.state = L.state;
                a.uin = L.uin;
                did |= 1;
            }
        }
        if (fz->kv_layer >= 0 && ps && !fz->ssq_out) {   // the row table shares the ssq scratch
            const LayerDesc& L = h->layer[fz->kv_layer];
            a.kv = 1;
            a.kv_H = L.param;
            a.kv_dh = h->cfg.head_dim;
            a.kv_in_cache = ps->kv_in_cache;
            a.kv_tmax = h->cfg.t_max;
            a.kv_C = ps->C;
            a.kv_T = ps->T;
            a.kv_base = h->kv_base;
            a.kc = (__nv_bfloat16*)L.kc;
            a.vc = (__nv_bfloat16*)L.vc;
            a.ks = (__nv_bfloat16*)L.ks;
            a.vs = (__nv_bfloat16*)L.vs;
            did |= 2;
        }
    }
    // The K/V-writing projection (an attention layer's QKV) starts once its predecessor has
    // ended instead of beside it. Started early, its 96 three-CTA clusters (12288 wide) were
    // placed piecemeal into the slots the predecessor freed, and the last one or two found no
    // GPC with room until CTAs of the launch itself finished: a 15 us tail at 13 token rows.
    const bool pdl = h->pdl != 0 && !(did & 2);
    if (!launch_tc(t, ta, tb, a, h->stream, pdl)) return false;
    if (fused) *fused = did;
    return true;
}

}  // namespace evs

// ---- projection without any allocation ------------------------------------------------------
// Same kernel, with its split-K scratch (partial sums, arrival counters, flag word) in one
// file-scope device array instead of a caller workspace. The array is fixed in size and
// resident on every GPU that loads the library until the process exits.
namespace evs {
namespace {

constexpr size_t kNoAllocPartFloats = (size_t)2 << 20;   // 8 MiB of fp32 partial sums
constexpr int kNoAllocCounters = 256;                    // 128-channel tiles: N <= 32768
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
    float part[kNoAllocPartFloats];
    int counters[kNoAllocCounters];
    uint32_t flags;
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

// Per-device set-up results: the array's device address and the kernel's shared-memory
// limit, filled once per device under the mutex (by the first call that finds them unset)
// and published through the atomic pointer after the limit is written.
std::mutex g_noalloc_mu;
std::atomic<NoAllocScratch*> g_noalloc_ptr[kNoAllocMaxDevices];
int g_noalloc_smem[kNoAllocMaxDevices];

// The current device's scratch address (set-up on first use), or null with *st set.
NoAllocScratch* noalloc_scratch(cudaStream_t s, evs_status* st, int* dev_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { *st = EVS_ERR_CUDA; return nullptr; }
    if (dev < 0 || dev >= kNoAllocMaxDevices) { *st = EVS_ERR_INVALID_ARG; return nullptr; }
    *dev_out = dev;
    NoAllocScratch* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p) return p;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    p = g_noalloc_ptr[dev].load(std::memory_order_relaxed);
    if (p) return p;
    // one-time set-up on this device (the device is current here): the array's address,
    // the kernel's shared-memory opt-in, and a cleared flag word
    if (cudaGetSymbolAddress((void**)&p, g_noalloc_scratch) != cudaSuccess || !p) {
        *st = EVS_ERR_CUDA;
        return nullptr;
    }
    const int smem_max = gemm_tc_init();
    if (smem_max < 0) { *st = EVS_ERR_CUDA; return nullptr; }
    if (cudaMemsetAsync(&p->flags, 0, sizeof(uint32_t), s) != cudaSuccess) { *st = EVS_ERR_CUDA; return nullptr; }
    g_noalloc_smem[dev] = smem_max;
    g_noalloc_ptr[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace
}  // namespace evs

extern "C" evs_status evs_projection_noalloc(const void* X, int32_t x_rows, const void* W, float* Y, int32_t M,
                                             int32_t N, int32_t K, int32_t ldy, int32_t accumulate,
                                             void* stream) {
    using namespace evs;
    if (!X || !W || !Y || !gemm_tc_supported(M, N, K) || x_rows < M || ldy < N) return EVS_ERR_INVALID_ARG;
    if (N / TC_BM > kNoAllocCounters) return EVS_ERR_CAPACITY;   // more channel tiles than counters
    cudaStream_t s = (cudaStream_t)stream;
    evs_status st = EVS_OK;
    int dev = -1;
    NoAllocScratch* sc = noalloc_scratch(s, &st, &dev);
    if (!sc) return st;
    // split-K partials always go through the fixed array here (no thread-block cluster);
    // the split count is capped so that every partial tile fits it (one split always does)
    const TcShape t = tc_shape(M, N, K, kNoAllocPartFloats, 1 << 30, /*allow_cluster=*/false);
    if (tc_part_floats(t, M, N) > kNoAllocPartFloats) return EVS_ERR_CAPACITY;
    CUtensorMap ta, tb;
    if (!make_map(&ta, W, (uint64_t)N, (uint64_t)K, TC_BM)) return EVS_ERR_CUDA;
    if (!make_map(&tb, X, (uint64_t)x_rows, (uint64_t)K, (uint32_t)(t.n_pad < 256 ? t.n_pad : 256))) return EVS_ERR_CUDA;
    if ((int)t.smem > g_noalloc_smem[dev]) return EVS_ERR_INVALID_ARG;
    // the array keeps the previous call's contents: the counters must start at zero
    if (cudaMemsetAsync(sc->counters, 0, sizeof(sc->counters), s) != cudaSuccess) return EVS_ERR_CUDA;
    TcArgs a{};
    a.Y = Y; a.ldy = ldy; a.M = M; a.N = N; a.kblocks = t.kblocks; a.splits = t.splits; a.n_pad = t.n_pad;
    a.stages = t.stages; a.accumulate = accumulate; a.ncols = t.ncols; a.kbs = t.kbs; a.cluster = t.cluster;
    a.part = sc->part; a.counters = sc->counters; a.flags = &sc->flags;
    if (!launch_tc(t, ta, tb, a, s, false)) return EVS_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? EVS_OK : EVS_ERR_CUDA;
}

extern "C" evs_status evs_projection_noalloc_flags(uint32_t* flags, int32_t clear, void* stream) {
    using namespace evs;
    if (!flags) return EVS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    evs_status st = EVS_OK;
    int dev = -1;
    NoAllocScratch* sc = noalloc_scratch(s, &st, &dev);
    if (!sc) return st;
    uint32_t v = 0;
    // a device-to-host copy into this stack word, then the stream is synchronised
    if (cudaMemcpyAsync(&v, &sc->flags, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return EVS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EVS_ERR_CUDA;
    *flags = v;
    if (clear && cudaMemsetAsync(&sc->flags, 0, sizeof(uint32_t), s) != cudaSuccess) return EVS_ERR_CUDA;
    return EVS_OK;
}
