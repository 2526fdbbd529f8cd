// Split-KV causal attention over the readable KV prefix on tcgen05 tensor cores.
//
// One CTA per (prefix chunk, sequence x head); the chunks are equal shares of the key tiles
// of the sequence's readable prefix, worked out from its length at run time. All queries of the sequence (every block
// position of every candidate: they share the prefix) are the N dimension of the MMAs, so
// each TMA-staged 128-key tile of K and V is read from HBM once and used by every query.
//   S^T[key][q] = K_tile . Q^T          (A = K tile, K-major; B = Q, K-major; D in TMEM)
//   softmax over the chunk, two passes  (max, then p = exp(s - m) and row sums)
//   O^T[dh][q] += V_tile^T . P_tile^T   (A = V tile read MN-major; B = P, K-major)
// The CTA writes unnormalised partials (o, m, l) per query; the combine kernel merges the
// chunks with the in-block causal keys.
//
// Warps 0-7 stage Q, run the softmax and the epilogue (warp w reads TMEM lanes
// 32(w%4)..32(w%4)+31; the two warpgroups share the query columns), warp 8 drives TMA,
// warp 9 issues the MMAs. dh = 128.
#include <cudaTypedefs.h>
#include <math.h>

#include "evs_common.cuh"
#include "sm100_ptx.cuh"

namespace evs {

constexpr int AT_KEYS = 128;                 // keys per tile (MMA M of the score product)
constexpr int AT_DH = 128;
constexpr int AT_TILE_BYTES = AT_KEYS * AT_DH * 2;   // 32 KiB: two 64-column swizzled halves
constexpr int AT_HALF = AT_TILE_BYTES / 2;

struct AttnArgs {
    const float* y;        // projection output, q in columns [head*dh, head*dh + dh)
    int ldy, H, Q, n_q;    // queries per sequence, padded to 16
    int tiles;             // key tiles per CTA (chunk = tiles * 128 keys)
    int splits, q_stride, stages, ncols;
    float scale;
    const int32_t* kv_base;
    float* part;           // [B][H][splits][q_stride][dh + 2]
    uint32_t* flags;
};

__device__ __forceinline__ uint32_t sw128_offset(int row, int col_elem) {
    // byte offset of bf16 element (row, col) inside a [rows][64] 128-byte-swizzled block
    return (uint32_t)row * 128u + ((uint32_t)((col_elem >> 3) ^ (row & 7)) << 4) + (uint32_t)(col_elem & 7) * 2u;
}

__global__ void __launch_bounds__(320, 2)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot[1];
    __shared__ volatile int abort_flag[1];
    __shared__ float red[4][128];
    __shared__ float m_sh[128], l_sh[128];

    pdl_trigger();
    pdl_wait();
    const int split = blockIdx.x, bh = blockIdx.y;
    const int b = bh / a.H, head = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.kv_base[b];
    // this CTA's equal share of the readable prefix's key tiles (at most a.tiles of them)
    const int nt_all = (n + AT_KEYS - 1) / AT_KEYS;
    const int t_lo = (int)((long long)nt_all * split / a.splits);
    const int t_hi = (int)((long long)nt_all * (split + 1) / a.splits);
    const int ntiles = min(t_hi - t_lo, a.tiles);
    const int k_lo = t_lo * AT_KEYS;
    const int k_hi = min(k_lo + ntiles * AT_KEYS, n);
    float* part = a.part + (((size_t)bh * a.splits + split) * a.q_stride) * (AT_DH + 2);

    if (ntiles == 0) {  // chunk past the readable prefix: empty partial
        for (int i = tid; i < a.Q; i += blockDim.x) {
            part[(size_t)i * (AT_DH + 2) + AT_DH] = -INFINITY;
            part[(size_t)i * (AT_DH + 2) + AT_DH + 1] = 0.f;
        }
        return;
    }

    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* ring = smem;                                            // [stages][2][128][128 B]
    uint8_t* sQ = ring + (size_t)a.stages * AT_TILE_BYTES;           // [2][n_q][128 B]
    uint8_t* sP = sQ + (size_t)2 * a.n_q * 128;                      // [tiles][2][n_q][128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(sP + (size_t)a.tiles * 2 * a.n_q * 128);
    uint64_t* empty = full + a.stages;
    uint64_t* s_done = empty + a.stages;
    uint64_t* p_ready = s_done + 1;
    uint64_t* o_done = p_ready + 1;

    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(s_done, 1);
        mbar_init(p_ready, 256);
        mbar_init(o_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(tmem_slot, (uint32_t)a.ncols);
        tmem_relinquish();
    }
    if (tid < 256) {  // stage Q (fp32 -> bf16, swizzled K-major), zero rows past Q
        const float* qsrc = a.y + (size_t)b * a.Q * a.ldy + (size_t)head * AT_DH;
        for (int e = tid; e < a.n_q * AT_DH; e += 256) {
            const int q = e / AT_DH, c = e % AT_DH;
            const float v = q < a.Q ? qsrc[(size_t)q * a.ldy + c] : 0.f;
            *reinterpret_cast<__nv_bfloat16*>(sQ + (size_t)(c >> 6) * a.n_q * 128 + sw128_offset(q, c & 63)) =
                __float2bfloat16_rn(v);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t o_col = (uint32_t)(a.tiles * a.n_q);

    if (warp == 8) {
        if (lane == 0) {  // ---- TMA: K tiles, then V tiles ---------------------------------
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < 2 * ntiles; ++i) {
                const int s = i % a.stages;
                const uint32_t ph = (uint32_t)(i / a.stages) & 1u;
                if (i >= a.stages && !mbar_wait(&empty[s], ph ^ 1u)) { *abort_flag = 1; break; }
                const CUtensorMap* m = i < ntiles ? &tmK : &tmV;
                const int row = k_lo + (i % ntiles) * AT_KEYS;
                uint8_t* dst = ring + (size_t)s * AT_TILE_BYTES;
                mbar_arrive_expect_tx(&full[s], (uint32_t)AT_TILE_BYTES);
                tma_load_3d(dst, m, 0, row, bh, &full[s], pol);
                tma_load_3d(dst + AT_HALF, m, 64, row, bh, &full[s], pol);
            }
        }
        __syncwarp();
    } else if (warp == 9) {
        if (lane == 0) {  // ---- MMA issuer ----------------------------------------------------
            const uint32_t id_s = idesc_bf16_f32(AT_KEYS, a.n_q);
            const uint32_t id_o = idesc_bf16_f32_amn(AT_DH, a.n_q);
            const uint32_t q0 = smem_u32(sQ);
            bool ok = true;
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t % a.stages;
                if (!mbar_wait(&full[s], (uint32_t)(t / a.stages) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t k0 = smem_u32(ring + (size_t)s * AT_TILE_BYTES);
#pragma unroll
                for (int kk = 0; kk < AT_DH / 16; ++kk) {
                    const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32u;
                    tc_mma_f16(tmem + (uint32_t)(t * a.n_q), smem_desc_sw128(k0 + half * AT_HALF + off),
                               smem_desc_sw128(q0 + half * (uint32_t)a.n_q * 128u + off), id_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(&empty[s]);
            }
            tc_commit(s_done);
            if (ok && !mbar_wait(p_ready, 0)) ok = false;
            tc_fence_after();
            for (int t = 0; t < ntiles && ok; ++t) {
                const int i = ntiles + t;
                const int s = i % a.stages;
                if (!mbar_wait(&full[s], (uint32_t)(i / a.stages) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t v0 = smem_u32(ring + (size_t)s * AT_TILE_BYTES);
                const uint32_t p0 = smem_u32(sP + (size_t)t * 2 * a.n_q * 128);
#pragma unroll
                for (int kk = 0; kk < AT_KEYS / 16; ++kk) {
                    const uint32_t half = (uint32_t)(kk >> 2), off = (uint32_t)(kk & 3) * 32u;
                    tc_mma_f16(tmem + o_col, smem_desc_sw128_mn(v0 + (uint32_t)kk * 16u * 128u, AT_HALF),
                               smem_desc_sw128(p0 + half * (uint32_t)a.n_q * 128u + off), id_o,
                               (t > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&empty[s]);
            }
            if (!ok) *abort_flag = 1;
            tc_commit(o_done);
        }
        __syncwarp();
    } else {
        // ---- softmax over the chunk: lane = key within a tile, columns = queries --------------
        // Eight warps: warp w reads TMEM lanes 32(w%4).., warpgroup w/4 takes half of the
        // 16-column query blocks. Scores go through exp2 with scale*log2(e) folded in.
        const int grp = warp >> 2, wq = warp & 3;
        const int nb = a.n_q / 16;
        const int split_b = nb >= 2 ? (nb + 1) / 2 : nb;
        const int g_lo = grp == 0 ? 0 : split_b * 16, g_hi = grp == 0 ? split_b * 16 : nb * 16;
        const float sl = a.scale * 1.4426950408889634f;
        const bool sok = mbar_wait(s_done, 0);
        tc_fence_after();
        const uint32_t trow = tmem + ((uint32_t)(wq * 32) << 16);
        const int row = wq * 32 + lane;
        for (int g = g_lo; g < g_hi; g += 16) {
            float mx[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) mx[j] = -INFINITY;
            for (int t = 0; t < ntiles; ++t) {
                float v[16];
                tmem_ld16(trow + (uint32_t)(t * a.n_q + g), v);
                if (k_lo + t * AT_KEYS + row < k_hi) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) mx[j] = fmaxf(mx[j], v[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float w = warp_max(mx[j]);
                if (lane == j) red[wq][g + j] = w;
            }
        }
        named_bar_sync(1, 256);
        for (int q = tid; q < a.n_q; q += 256)   // raw-score max; scale > 0 keeps the order
            m_sh[q] = fmaxf(fmaxf(red[0][q], red[1][q]), fmaxf(red[2][q], red[3][q])) * sl;
        named_bar_sync(1, 256);
        for (int g = g_lo; g < g_hi; g += 16) {
            float sum[16], mq[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) { sum[j] = 0.f; mq[j] = m_sh[g + j]; }
            for (int t = 0; t < ntiles; ++t) {
                float v[16];
                tmem_ld16(trow + (uint32_t)(t * a.n_q + g), v);
                const bool valid = k_lo + t * AT_KEYS + row < k_hi;
                uint8_t* pt = sP + (size_t)t * 2 * a.n_q * 128 + (size_t)(row >> 6) * a.n_q * 128;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float p = valid ? ex2_approx(fmaf(v[j], sl, -mq[j])) : 0.f;
                    const __nv_bfloat16 pb = __float2bfloat16_rn(p);
                    sum[j] += __bfloat162float(pb);   // normalise by what the MMA multiplies
                    *reinterpret_cast<__nv_bfloat16*>(pt + sw128_offset(g + j, row & 63)) = pb;
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float w = warp_sum(sum[j]);
                if (lane == j) red[wq][g + j] = w;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 256);
        for (int q = tid; q < a.n_q; q += 256) l_sh[q] = red[0][q] + red[1][q] + red[2][q] + red[3][q];
        mbar_arrive(p_ready);
        // ---- epilogue: lane = dh index, columns = queries --------------------------------------
        const bool ook = mbar_wait(o_done, 0);
        tc_fence_after();
        const bool bad = !sok || !ook || *abort_flag;
        if (bad && tid == 0) atomicOr(a.flags, (uint32_t)EVS_FLAG_TIMEOUT);
        named_bar_sync(1, 256);
        for (int g = g_lo; g < g_hi; g += 16) {
            float v[16];
            tmem_ld16(trow + o_col + (uint32_t)g, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int q = g + j;
                if (q < a.Q && !bad) part[(size_t)q * (AT_DH + 2) + row] = v[j];
            }
        }
        // m in natural units of the scaled score (the combine's convention)
        for (int q = tid; q < a.Q; q += 256) {
            part[(size_t)q * (AT_DH + 2) + AT_DH] = bad ? -INFINITY : m_sh[q] * 0.6931471805599453f;
            part[(size_t)q * (AT_DH + 2) + AT_DH + 1] = bad ? 0.f : l_sh[q];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)a.ncols);
    }
}

// ---- host side ------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
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

// KV cache [B*H][t_max][128] bf16 as a 3-D map with a 64 x 128-key box, 128-byte swizzle.
bool make_kv_map(CUtensorMap* m, const void* base, int t_max, int bh) {
    auto fn = attn_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)AT_DH, (cuuint64_t)t_max, (cuuint64_t)bh};
    const cuuint64_t strides[2] = {(cuuint64_t)AT_DH * 2, (cuuint64_t)t_max * AT_DH * 2};
    const cuuint32_t box[3] = {64, AT_KEYS, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Chunking of the prefix for a pass with Q queries per sequence (dh = 128, bf16).
AttnPlan attn_tc_plan(int Q, int B, int H, int t_max, int smem_max) {
    if (Q > 16) {   // many queries: the streaming kernel with one query per TMEM lane
        const AttnPlan f = attn_fa_plan(Q, B, H, t_max, smem_max);
        if (f.ok) return f;
    }
    AttnPlan p{};
    p.n_q = (Q + 15) / 16 * 16;
    if (Q < 1 || p.n_q > 128) return p;
    // tiles per CTA bounded by TMEM (S tiles + O <= 512 columns) and by the P buffer
    int tmax = 512 / p.n_q - 1;
    const int p_cap = (96 * 1024) / (p.n_q * 256);
    if (tmax > p_cap) tmax = p_cap;
    if (tmax > 16) tmax = 16;
    if (tmax < 1) return p;
    // Chunks are dealt out at run time in equal shares of the readable prefix (see the
    // kernel), so the plan fixes only the number of splits and the largest share. Prefer one
    // wave of two CTAs per SM (TMEM and shared memory permitting); past tmax tiles per CTA,
    // as many splits of tmax tiles as the cache needs.
    const long long total_tiles = (t_max + AT_KEYS - 1) / AT_KEYS;
    const long long bh = (long long)B * H;
    auto fits_two = [&](long long per) {
        const long long fixed = 1024 + 2LL * p.n_q * 128 + per * 2 * p.n_q * 128 + 64 * 8;
        return (per + 1) * p.n_q <= 256 && fixed + 2LL * AT_TILE_BYTES <= 110 * 1024;
    };
    long long splits = 304 / bh;
    if (splits < 1) splits = 1;
    long long per = (total_tiles + splits - 1) / splits;
    if (per <= tmax && !fits_two(per)) {          // one wave of one CTA per SM instead
        splits = 152 / bh;
        if (splits < 1) splits = 1;
        per = (total_tiles + splits - 1) / splits;
    }
    if (per > tmax) {
        per = tmax;
        splits = (total_tiles + per - 1) / per;
    }
    p.tiles = (int)per;
    p.splits = (int)splits;
    int need = (p.tiles + 1) * p.n_q;
    p.ncols = 32;
    while (p.ncols < need) p.ncols <<= 1;
    // ring of 32 KiB stages in what is left of shared memory
    const int fixed = 1024 + 2 * p.n_q * 128 + p.tiles * 2 * p.n_q * 128 + 64 * 8;
    // keep two CTAs per SM when the chunk allows it, so one CTA's start-up and softmax
    // overlap another's streaming
    const int budget = fixed + 2 * AT_TILE_BYTES <= 110 * 1024 ? 110 * 1024 : smem_max;
    p.stages = (budget - fixed) / AT_TILE_BYTES;
    if (p.stages > 4) p.stages = 4;
    if (p.stages > 2 * p.tiles) p.stages = 2 * p.tiles;
    if (p.stages < 2) { p.n_q = 0; return p; }
    p.smem = fixed + p.stages * AT_TILE_BYTES;
    p.ok = 1;
    return p;
}

int attn_tc_init() {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, attn_tc_kernel) != cudaSuccess)
        return -1;
    const int dyn = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
        return -1;
    return dyn;
}

bool launch_attn_tc(evs_handle* h, int li, const Pass& p, const AttnPlan& plan) {
    if (plan.fa) return launch_attn_fa(h, li, p, plan);
    const LayerDesc& L = h->layer[li];
    const int H = L.param;
    CUtensorMap tk, tv;
    if (!make_kv_map(&tk, L.kc, h->cfg.t_max, p.B * H) || !make_kv_map(&tv, L.vc, h->cfg.t_max, p.B * H))
        return false;
    AttnArgs a{h->y, 3 * h->cfg.d, H, p.C * p.T, plan.n_q, plan.tiles, plan.splits, h->g.q_max, plan.stages,
               plan.ncols, 1.0f / sqrtf((float)AT_DH), h->kv_base, h->attn_part, h->flags};
    return launch_k(h, attn_tc_kernel, dim3(plan.splits, p.B * H), dim3(320), (size_t)plan.smem, tk, tv, a) ==
           cudaSuccess;
}

}  // namespace evs
