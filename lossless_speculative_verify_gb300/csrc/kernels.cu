// Block-forward, acceptance and slicing kernels (CUDA cores), sm_103a.
//
// Steps of one verification round (EvSpark summary, Figure 1(c)-(d)): embed the block
// [anchor, d_1..d_gamma]; per layer RMS-normalise, project, run the mixer (depthwise FIR
// over [cached tail || block inputs], modal IIR scan keeping every s_t, or causal
// attention over the readable prefix plus the in-block keys), project back into the
// residual; then logits, acceptance, and slicing the state at the accepted index k.
#include "evs_common.cuh"

namespace evs {

// =========================================================================================
// embedding gather; records the pass's starting KV length
// =========================================================================================
template <typename T>
__global__ void embed_kernel(const T* __restrict__ E, const int32_t* __restrict__ tokens,
                             int tok_stride_bc, const int32_t* __restrict__ anchor,
                             float* __restrict__ h, int d, int C, int Tb, int vocab, int B,
                             const int32_t* __restrict__ kv_len, int32_t* __restrict__ kv_base,
                             uint32_t* __restrict__ flags, __nv_bfloat16* __restrict__ hb,
                             float* __restrict__ ssq, int ssq_tiles, int ssq_ld) {
    __shared__ float red[32];
    pdl_trigger();
    pdl_wait();
    const int m = blockIdx.x;
    const int bc = m / Tb, i = m % Tb, b = bc / C;
    int tok = (i == 0 && anchor != nullptr) ? anchor[b] : tokens[(size_t)bc * tok_stride_bc + i];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) atomicOr(flags, (uint32_t)EVS_FLAG_BAD_TOKEN);
        tok = tok < 0 ? 0 : vocab - 1;
    }
    const T* row = E + (size_t)tok * d;
    float* out = h + (size_t)m * d;
    float ss = 0.f;
    // eight consecutive channels a thread (d is a multiple of 64): 16- or 32-byte loads, two
    // 16-byte stores of h and one of bf16(h)
    for (int c = 8 * threadIdx.x; c < d; c += 8 * blockDim.x) {
        float v[8];
        if constexpr (sizeof(T) == 2) {
            const uint4 raw = *reinterpret_cast<const uint4*>(row + c);
            const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(p2[k]);
                v[2 * k] = f.x;
                v[2 * k + 1] = f.y;
            }
        } else {
            const float4 a = *reinterpret_cast<const float4*>(row + c), b4 = *reinterpret_cast<const float4*>(row + c + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b4.x; v[5] = b4.y; v[6] = b4.z; v[7] = b4.w;
        }
        *reinterpret_cast<float4*>(out + c) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4*>(out + c + 4) = make_float4(v[4], v[5], v[6], v[7]);
#pragma unroll
        for (int k = 0; k < 8; ++k) ss += v[k] * v[k];
        if (hb) {
            uint4 pk;
            __nv_bfloat162* q2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
            for (int k = 0; k < 4; ++k) q2[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            *reinterpret_cast<uint4*>(hb + (size_t)m * d + c) = pk;
        }
    }
    if (ssq) {  // the row's sum of squares in tile slot 0, the other slots cleared
        ss = block_sum(ss, red);
        for (int t = threadIdx.x; t < ssq_tiles; t += blockDim.x) ssq[(size_t)t * ssq_ld + m] = t == 0 ? ss : 0.f;
    }
    if (m == 0)
        for (int j = threadIdx.x; j < B; j += blockDim.x) kv_base[j] = kv_len[j];
}

// =========================================================================================
// RMS norm (no gain): act = h / sqrt(mean(h^2) + eps), stored in the projection dtype
// =========================================================================================
template <typename T>
__global__ void rmsnorm_kernel(const float* __restrict__ h, T* __restrict__ out, int d) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[32];
    const int m = blockIdx.x;
    const float* row = h + (size_t)m * d;
    float ss = 0.f;
    for (int c = threadIdx.x; c < d; c += blockDim.x) ss += row[c] * row[c];
    ss = block_sum(ss, red);
    const float r = rsqrtf(ss / (float)d + 1e-6f);
    T* o = out + (size_t)m * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) o[c] = from_f32<T>(row[c] * r);
}

// =========================================================================================
// CUDA-core projection: Y[m][n] (+)= sum_k A[m][k] * W[n][k]   (W out-major)
// =========================================================================================
constexpr int GS_BM = 16, GS_BN = 64, GS_BK = 32;

template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ A, const T* __restrict__ W,
                                                        float* __restrict__ Y, int M, int N, int K,
                                                        int ldy, int accumulate) {
    pdl_trigger();
    pdl_wait();
    __shared__ float As[GS_BM][GS_BK + 1];
    __shared__ float Ws[GS_BN][GS_BK + 1];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * GS_BM, n0 = blockIdx.x * GS_BN;
    const int r = tid / 16, c0 = (tid % 16) * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += GS_BK) {
        for (int e = tid; e < GS_BM * GS_BK; e += 256) {
            const int rr = e / GS_BK, kk = e % GS_BK;
            const int m = m0 + rr;
            As[rr][kk] = (m < M && k0 + kk < K) ? to_f32(A[(size_t)m * K + k0 + kk]) : 0.f;
        }
        for (int e = tid; e < GS_BN * GS_BK; e += 256) {
            const int rr = e / GS_BK, kk = e % GS_BK;
            const int n = n0 + rr;
            Ws[rr][kk] = (n < N && k0 + kk < K) ? to_f32(W[(size_t)n * K + k0 + kk]) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < GS_BK; ++kk) {
            const float a = As[r][kk];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = fmaf(a, Ws[c0 + j][kk], acc[j]);
        }
        __syncthreads();
    }
    const int m = m0 + r;
    if (m >= M) return;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int n = n0 + c0 + j;
        if (n >= N) continue;
        float* dst = Y + (size_t)m * ldy + n;
        *dst = accumulate ? (*dst + acc[j]) : acc[j];
    }
}

// =========================================================================================
// Depthwise FIR over [cached tail || block inputs]: y_t = sum_{j<L} taps[c][j] v_{t-j}.
// One thread per (sequence-candidate, channel); loads coalesced along the channel.
// =========================================================================================
template <typename T>
__global__ void fir_kernel(const float* __restrict__ Y, int ldy, T* __restrict__ out, int d,
                           int C, int Tb, int commit, const float* __restrict__ taps, int L,
                           float* __restrict__ tail, float* __restrict__ stage) {
    pdl_trigger();
    pdl_wait();
    const int ch = blockIdx.x * blockDim.x + threadIdx.x;
    const int bc = blockIdx.y, b = bc / C;
    if (ch >= d) return;
    // w[j] taps; hist[j] = x_{t-1-j}, the newest input first (fixed register indices)
    float w[16], hist[15];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = (j < L) ? taps[(size_t)ch * L + j] : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) hist[j] = (j < L - 1) ? tail[((size_t)b * (L - 1) + (L - 2 - j)) * d + ch] : 0.f;
    const int srows = L - 1 + Tb;
    float* st = stage + (size_t)bc * srows * d;
    if (!commit) {
#pragma unroll
        for (int j = 0; j < 15; ++j)
            if (j < L - 1) st[(size_t)(L - 2 - j) * d + ch] = hist[j];
    }
    for (int i0 = 0; i0 < Tb; i0 += 8) {
        float vin[8];   // eight positions' inputs requested before any is used
#pragma unroll
        for (int u = 0; u < 8; ++u)
            vin[u] = (i0 + u < Tb) ? Y[((size_t)bc * Tb + i0 + u) * ldy + ch] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            if (i < Tb) {
                const size_t m = (size_t)bc * Tb + i;
                const float v = vin[u];
                float y = w[0] * v;
#pragma unroll
                for (int j = 1; j < 16; ++j)
                    if (j < L) y = fmaf(w[j], hist[j - 1], y);
#pragma unroll
                for (int j = 14; j > 0; --j) hist[j] = hist[j - 1];
                hist[0] = v;
                out[m * d + ch] = from_f32<T>(y);
                if (!commit) st[(size_t)(L - 1 + i) * d + ch] = v;
            }
        }
    }
    if (commit) {
#pragma unroll
        for (int j = 0; j < 15; ++j)
            if (j < L - 1) tail[((size_t)b * (L - 1) + (L - 2 - j)) * d + ch] = hist[j];
    }
}

// =========================================================================================
// Modal IIR scan s_t = lam * s_{t-1} + b * u_t, y_t = Re sum_n c_n s_{t,n}.
// N consecutive lanes hold the N poles of one channel; y by a shuffle reduction.
// A prefill pass (commit) leaves the last s_t in the state. A verify pass writes no state:
// its inputs u_t stay where the in-projection put them, and slicing recomputes s_k.
// =========================================================================================
template <typename T, int NP>   // NP: poles per channel when fixed at compile time, else 0
__global__ void __launch_bounds__(256) iir_kernel(const float* __restrict__ Y, int ldy, T* __restrict__ out, int d,
                                                  int Nrt, int C, int Tb, int commit, const float2* __restrict__ lam,
                                                  const float2* __restrict__ bb, const float2* __restrict__ cc,
                                                  float2* __restrict__ state) {
    pdl_trigger();
    pdl_wait();
    const int N = NP > 0 ? NP : Nrt;
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    const int bc = blockIdx.y, b = bc / C;
    if (g >= d * N) return;  // d*N is a multiple of 32: whole warps leave together
    const int ch = g / N, n = g % N;
    const float2 l = lam[g], bq = bb[g], cq = cc[g];
    float2 s = state[(size_t)b * d * N + g];
    const float* yin = Y + (size_t)bc * Tb * ldy + ch;
    T* op = out + (size_t)bc * Tb * d + ch;
    for (int i0 = 0; i0 < Tb; i0 += 8) {
        // eight positions: inputs requested together, the recurrence, then the eight
        // readouts reduced over the pole lanes side by side
        float uin[8], q[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) uin[k] = (i0 + k < Tb) ? yin[(size_t)(i0 + k) * ldy] : 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (i0 + k < Tb) {
                const float u = uin[k];
                s = make_float2(fmaf(l.x, s.x, fmaf(-l.y, s.y, bq.x * u)), fmaf(l.x, s.y, fmaf(l.y, s.x, bq.y * u)));
            }
            q[k] = fmaf(cq.x, s.x, -cq.y * s.y);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            if (o < N) {
#pragma unroll
                for (int k = 0; k < 8; ++k) q[k] += __shfl_xor_sync(0xffffffffu, q[k], o);
            }
        }
        if (n == 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (i0 + k < Tb) op[(size_t)(i0 + k) * d] = from_f32<T>(q[k]);
        }
    }
    if (commit) state[(size_t)b * d * N + g] = s;
}

// The same scan with four poles per thread (N/4 lanes per channel): the readout needs only
// log2(N/4) shuffle levels. With 16 bf16 poles, four CTAs an SM (64 registers, no spills): 1024
// CTAs at 4 x 4 candidates take 1.7 waves instead of 2.2 (-1.7 us per round).
template <typename T, int NP>
__global__ void __launch_bounds__(256, (NP == 16 && sizeof(T) == 2) ? 4 : 2)
    iir_quad_kernel(const float* __restrict__ Y, int ldy, T* __restrict__ out, int d, int C, int Tb, int commit,
                    const float2* __restrict__ lam, const float2* __restrict__ bb, const float2* __restrict__ cc,
                    float2* __restrict__ state) {
    constexpr int PPT = NP < 4 ? NP : 4;     // poles per thread
    constexpr int LPC = NP / PPT;            // lanes per channel
    pdl_trigger();
    pdl_wait();
    const int g = blockIdx.x * blockDim.x + threadIdx.x;
    const int bc = blockIdx.y, b = bc / C;
    if (g >= d * LPC) return;   // d*LPC is a multiple of 32 here: whole warps leave together
    const int ch = g / LPC, k0 = (g % LPC) * PPT;
    float2 l[PPT], bq[PPT], cq[PPT], s[PPT];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        l[k] = lam[(size_t)ch * NP + k0 + k];
        bq[k] = bb[(size_t)ch * NP + k0 + k];
        cq[k] = cc[(size_t)ch * NP + k0 + k];
        s[k] = state[((size_t)b * d + ch) * NP + k0 + k];
    }
    const float* yin = Y + (size_t)bc * Tb * ldy + ch;
    for (int i0 = 0; i0 < Tb; i0 += 8) {
        float uin[8], q[8];   // eight positions' inputs requested before any is used
#pragma unroll
        for (int u = 0; u < 8; ++u) uin[u] = (i0 + u < Tb) ? yin[(size_t)(i0 + u) * ldy] : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            float y = 0.f;
            if (i0 + u < Tb) {
#pragma unroll
                for (int k = 0; k < PPT; ++k) {
                    s[k] = make_float2(fmaf(l[k].x, s[k].x, fmaf(-l[k].y, s[k].y, bq[k].x * uin[u])),
                                       fmaf(l[k].x, s[k].y, fmaf(l[k].y, s[k].x, bq[k].y * uin[u])));
                    y = fmaf(cq[k].x, s[k].x, fmaf(-cq[k].y, s[k].y, y));
                }
            }
            q[u] = y;
        }
#pragma unroll
        for (int o = LPC / 2; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 8; ++u) q[u] += __shfl_xor_sync(0xffffffffu, q[u], o);
        if (k0 == 0) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i0 + u < Tb) out[((size_t)bc * Tb + i0 + u) * d + ch] = from_f32<T>(q[u]);
        }
    }
    if (commit) {
#pragma unroll
        for (int k = 0; k < PPT; ++k) state[((size_t)b * d + ch) * NP + k0 + k] = s[k];
    }
}

// =========================================================================================
// Block K/V rows from the fused QKV projection output into the cache (one candidate)
// or the per-candidate side buffer.
// =========================================================================================
template <typename T>
__global__ void kv_write_kernel(const float* __restrict__ Y, int ldy, int d, int H, int dh, int C,
                                int Tb, int in_cache, int t_max, const int32_t* __restrict__ kv_base,
                                T* __restrict__ kc, T* __restrict__ vc, T* __restrict__ ks,
                                T* __restrict__ vs, uint32_t* __restrict__ flags) {
    pdl_trigger();
    pdl_wait();
    const int m = blockIdx.y;
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= d) return;
    const int bc = m / Tb, i = m % Tb, b = bc / C;
    const int hh = col / dh, e = col % dh;
    const float kval = Y[(size_t)m * ldy + d + col];
    const float vval = Y[(size_t)m * ldy + 2 * d + col];
    if (in_cache) {
        const int t = kv_base[b] + i;
        if (t >= t_max) {
            if (col == 0) atomicOr(flags, (uint32_t)EVS_FLAG_KV_OVERFLOW);
            return;
        }
        const size_t o = (((size_t)b * H + hh) * t_max + t) * dh + e;
        kc[o] = from_f32<T>(kval);
        vc[o] = from_f32<T>(vval);
    } else {
        const size_t o = (((size_t)bc * H + hh) * Tb + i) * dh + e;
        ks[o] = from_f32<T>(kval);
        vs[o] = from_f32<T>(vval);
    }
}

// =========================================================================================
// Split-KV attention over the readable prefix (CUDA cores). One CTA per (split, sequence x
// head, group of 16 queries). Writes unnormalised partial (o, m, l) per query.
// =========================================================================================
constexpr int AQ = 16, AK = 64;

template <typename T>
__global__ void __launch_bounds__(256) attn_split_kernel(
    const float* __restrict__ Y, int ldy, const T* __restrict__ kc, const T* __restrict__ vc, int H,
    int dh, int Q, int q_max, int t_max, int chunk, int splits, const int32_t* __restrict__ kv_base,
    float* __restrict__ part) {
    pdl_trigger();
    pdl_wait();
    __shared__ float qs[AQ][128];
    __shared__ float kvs[AK][129];
    __shared__ float ps[AQ][AK];
    __shared__ float row_m[AQ], row_l[AQ], row_scale[AQ];
    const int s = blockIdx.x, bh = blockIdx.y, b = bh / H, hh = bh % H;
    const int q0 = blockIdx.z * AQ;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = kv_base[b];
    const int k_lo = s * chunk, k_hi = min(k_lo + chunk, n);
    const float scale = rsqrtf((float)dh);
    for (int e = tid; e < AQ * dh; e += 256) {
        const int r = e / dh, c = e % dh;
        const int qi = q0 + r;
        qs[r][c] = (qi < Q) ? Y[((size_t)b * Q + qi) * ldy + hh * dh + c] * scale : 0.f;
    }
    if (tid < AQ) { row_m[tid] = -INFINITY; row_l[tid] = 0.f; }
    // thread -> 8 outputs of O: row tid / 16, columns (tid % 16) + 16 * u
    const int orow = tid / 16, ocol = tid % 16;
    float o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = 0.f;
    const T* kbase = kc + ((size_t)b * H + hh) * t_max * dh;
    const T* vbase = vc + ((size_t)b * H + hh) * t_max * dh;
    __syncthreads();
    for (int t0 = k_lo; t0 < k_hi; t0 += AK) {
        const int nk = min(AK, k_hi - t0);
        for (int e = tid; e < AK * dh; e += 256) {
            const int r = e / dh, c = e % dh;
            kvs[r][c] = (r < nk) ? to_f32(kbase[(size_t)(t0 + r) * dh + c]) : 0.f;
        }
        __syncthreads();
        {   // scores: thread -> query tid/16, keys (tid%16) + 16u
            const int r = tid / 16;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = (tid % 16) + 16 * u;
                float acc = 0.f;
                for (int c = 0; c < dh; ++c) acc = fmaf(qs[r][c], kvs[j][c], acc);
                ps[r][j] = (j < nk) ? acc : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax: warp w owns query rows 2w, 2w+1
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = warp * 2 + rr;
            const float a = ps[r][lane], c2 = ps[r][lane + 32];
            const float tmax = warp_max(fmaxf(a, c2));
            const float m_old = row_m[r];
            const float m_new = fmaxf(m_old, tmax);
            const float pa = (a == -INFINITY) ? 0.f : __expf(a - m_new);
            const float pb = (c2 == -INFINITY) ? 0.f : __expf(c2 - m_new);
            const float tsum = warp_sum(pa + pb);
            ps[r][lane] = pa;
            ps[r][lane + 32] = pb;
            __syncwarp();
            if (lane == 0) {
                const float sc = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
                row_scale[r] = sc;
                row_l[r] = row_l[r] * sc + tsum;
                row_m[r] = m_new;
            }
        }
        __syncthreads();
        for (int e = tid; e < AK * dh; e += 256) {
            const int r = e / dh, c = e % dh;
            kvs[r][c] = (r < nk) ? to_f32(vbase[(size_t)(t0 + r) * dh + c]) : 0.f;
        }
        __syncthreads();
        {
            const float sc = row_scale[orow];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int c = ocol + 16 * u;
                if (c < dh) {
                    float acc = o[u] * sc;
                    for (int j = 0; j < nk; ++j) acc = fmaf(ps[orow][j], kvs[j][c], acc);
                    o[u] = acc;
                }
            }
        }
        __syncthreads();
    }
    const int qi = q0 + orow;
    if (qi < Q) {
        float* dst = part + ((((size_t)b * H + hh) * splits + s) * q_max + qi) * (dh + 2);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = ocol + 16 * u;
            if (c < dh) dst[c] = o[u];
        }
        if (ocol == 0) { dst[dh] = row_m[orow]; dst[dh + 1] = row_l[orow]; }
    }
}

// Merge the prefix partials with the in-block causal keys of the query's own candidate,
// normalise, and store o in the projection dtype. One CTA (four warps) per (sequence x head,
// candidate, four consecutive block positions), a warp per query; lanes own dh/32 output
// columns. The partials are folded PB chunks at a time (every load of a batch in flight
// before any is used) with a running maximum; then the in-block keys j <= i, staged
// 32 rows at a time in shared memory, one score per lane, the same way. dh is 16..128.
constexpr int CMB_ROWS = 32;
constexpr int CMB_DHMAX = 128;

// PB = 4 leaves registers for five bf16 CTAs an SM, for grids of several waves; PB = 8 takes
// one round trip fewer where five or six chunks meet a query.
template <typename T, int EPL, int PB>
__global__ void __launch_bounds__(128, (PB == 4 && sizeof(T) == 2) ? 5 : 4) attn_combine_kernel(
    const float* __restrict__ Y, int ldy, const T* __restrict__ kc, const T* __restrict__ vc,
    const T* __restrict__ ks, const T* __restrict__ vs, int H, int dh, int C, int Tb, int Q, int q_max,
    int t_max, int splits, int chunk, int B, int fa_grid, int in_cache, const int32_t* __restrict__ kv_base,
    const float* __restrict__ part, T* __restrict__ out, int d) {
    // dependents launch only once the attention partials are complete: an output projection
    // starting earlier would stream its weights against the attention kernel's K / V reads
    pdl_wait();
    pdl_trigger();
    // in-block rows in the cache dtype (small enough to share an SM with the attention
    // kernel, so the launch can start early); key rows padded so one key per lane is
    // conflict-free
    __shared__ T k_s[CMB_ROWS][CMB_DHMAX + 2];
    __shared__ __align__(16) T v_s[CMB_ROWS][CMB_DHMAX];
    __shared__ float q_s[4][CMB_DHMAX];
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, hh = bh % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = blockIdx.z * 4, i = i0 + warp;
    const int i_end = min(i0 + 4, Tb);                   // queries of this CTA: [i0, i_end)
    const bool live = i < Tb;
    const int qi = c * Tb + i;
    const int n = kv_base[b];  // rows n + j past t_max were never written (overflow flag set);
                               // their reads are clamped to stay in bounds
    // partial slots of this (sequence, head): chunk > 0, fixed chunks of the prefix (the first
    // ceil(n / chunk) slots); fa_grid > 0, the persistent tensor-core kernel's runs of key tiles
    // laid end to end over fa_grid CTAs (one slot per CTA whose run meets this prefix)
    int used = chunk > 0 ? min((n + chunk - 1) / chunk, splits) : splits;
    if (fa_grid > 0) {
        long long total = 0, start = 0;
        int ntb = 0;
        for (int bb = 0; bb < B; ++bb) {
            const int nt = (kv_base[bb] + 127) / 128;
            if (bb < b) start += (long long)H * nt;
            if (bb == b) ntb = nt;
            total += (long long)H * nt;
        }
        start += (long long)hh * ntb;
        used = 0;
        if (ntb > 0) {
            const long long W = (total + fa_grid - 1) / fa_grid;
            used = (int)((start + ntb - 1) / W - start / W + 1);
        }
        used = min(used, splits);
    }
    const float scale = rsqrtf((float)dh);
    const int e0 = lane * EPL;
    const bool act = e0 < dh;
    // issue the query row and the first in-block rows' loads together, then store them
    float qv[CMB_DHMAX / 32];
#pragma unroll
    for (int u = 0; u < CMB_DHMAX / 32; ++u) {
        const int e = lane + 32 * u;
        qv[u] = (live && e < dh) ? Y[((size_t)b * Q + qi) * ldy + hh * dh + e] : 0.f;
    }
    constexpr int PE = 16 / sizeof(T);                   // elements per 16-byte piece
    constexpr int MAXP = CMB_ROWS * CMB_DHMAX / PE / 128;
    const int per_row = dh / PE;
    uint4 kr4[MAXP], vr4[MAXP];
    auto stage_load = [&](int j0, int jn) {
#pragma unroll
        for (int u = 0; u < MAXP; ++u) {
            const int idx = tid + 128 * u;
            if (idx < jn * per_row) {
                const int jj = idx / per_row, e = (idx % per_row) * PE, j = j0 + jj;
                const size_t kr = in_cache ? (((size_t)b * H + hh) * t_max + min(n + j, t_max - 1)) * dh
                                           : ((((size_t)(b * C + c)) * H + hh) * Tb + j) * dh;
                kr4[u] = *reinterpret_cast<const uint4*>((in_cache ? kc : ks) + kr + e);
                vr4[u] = *reinterpret_cast<const uint4*>((in_cache ? vc : vs) + kr + e);
            }
        }
    };
    auto stage_store = [&](int jn) {
#pragma unroll
        for (int u = 0; u < MAXP; ++u) {
            const int idx = tid + 128 * u;
            if (idx < jn * per_row) {
                const int jj = idx / per_row, e = (idx % per_row) * PE;
                const T* kp = reinterpret_cast<const T*>(&kr4[u]);
#pragma unroll
                for (int x = 0; x < PE; ++x) k_s[jj][e + x] = kp[x];
                *reinterpret_cast<uint4*>(&v_s[jj][e]) = vr4[u];
            }
        }
    };
    stage_load(0, min(CMB_ROWS, i_end));
    float M = -INFINITY, L = 0.f, O[EPL];
#pragma unroll
    for (int u = 0; u < EPL; ++u) O[u] = 0.f;
    // fold a batch with maximum mb: rescale what is summed when the running maximum moves
    auto rebase = [&](float mb) {
        if (mb > M) {
            const float f = M == -INFINITY ? 0.f : __expf(M - mb);
            L *= f;
#pragma unroll
            for (int u = 0; u < EPL; ++u) O[u] *= f;
            M = mb;
        }
    };
    if (live) {
        const float* pq = part + ((size_t)bh * splits * q_max + qi) * (dh + 2);
        const size_t pstride = (size_t)q_max * (dh + 2);
        for (int s0 = 0; s0 < used; s0 += PB) {
            float ms[PB], ls[PB], os[PB][EPL];
#pragma unroll
            for (int j = 0; j < PB; ++j) {
                const bool on = s0 + j < used;
                ms[j] = on ? pq[(s0 + j) * pstride + dh] : -INFINITY;
                ls[j] = on ? pq[(s0 + j) * pstride + dh + 1] : 0.f;
#pragma unroll
                for (int u = 0; u < EPL; ++u) os[j][u] = (on && act) ? pq[(s0 + j) * pstride + e0 + u] : 0.f;
            }
            float mb = -INFINITY;
#pragma unroll
            for (int j = 0; j < PB; ++j) mb = fmaxf(mb, ms[j]);
            if (mb == -INFINITY) continue;        // empty chunks only
            rebase(mb);
#pragma unroll
            for (int j = 0; j < PB; ++j) {
                if (ms[j] == -INFINITY) continue;  // an empty chunk leaves its o unwritten
                const float w = __expf(ms[j] - M);
                L = fmaf(ls[j], w, L);
#pragma unroll
                for (int u = 0; u < EPL; ++u) O[u] = fmaf(os[j][u], w, O[u]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < CMB_DHMAX / 32; ++u)
        if (lane + 32 * u < dh) q_s[warp][lane + 32 * u] = qv[u];
    stage_store(min(CMB_ROWS, i_end));
    // in-block keys j <= i, 32 staged rows at a time (the CTA's queries see keys < i_end);
    // the first rows were staged above
    for (int j0 = 0; j0 < i_end; j0 += CMB_ROWS) {
        const int jn = min(CMB_ROWS, i_end - j0);
        if (j0 > 0) {
            __syncthreads();                      // the previous rows are no longer read
            stage_load(j0, jn);
            stage_store(jn);
        }
        __syncthreads();
        if (!live || j0 > i) continue;
        const int jhi = min(jn - 1, i - j0);      // last staged key this query sees
        float sc = -INFINITY;
        if (lane <= jhi) {
            float acc = 0.f;
            for (int e = 0; e < dh; ++e) acc = fmaf(q_s[warp][e], to_f32(k_s[lane][e]), acc);
            sc = acc * scale;
        }
        rebase(warp_max(sc));
        const float w = lane <= jhi ? __expf(sc - M) : 0.f;
        L += warp_sum(w);
        for (int jj = 0; jj <= jhi; ++jj) {
            const float wj = __shfl_sync(0xffffffffu, w, jj);
#pragma unroll
            for (int u = 0; u < EPL; ++u)
                if (act) O[u] = fmaf(wj, to_f32(v_s[jj][e0 + u]), O[u]);
        }
    }
    if (live && act) {
        const float inv = 1.f / L;
#pragma unroll
        for (int u = 0; u < EPL; ++u) out[((size_t)b * Q + qi) * d + hh * dh + e0 + u] = from_f32<T>(O[u] * inv);
    }
}

// =========================================================================================
// Softmax + acceptance. One CTA (256 threads) per sequence; candidates in turn.
// =========================================================================================
constexpr int ACC_THREADS = 256;

struct ArgMax { float v; int i; };

__device__ __forceinline__ ArgMax better(ArgMax a, ArgMax b) {
    if (b.v > a.v || (b.v == a.v && b.i < a.i)) return b;
    return a;
}

__device__ ArgMax block_argmax(ArgMax a, float* redv, int* redi) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax t{__shfl_xor_sync(0xffffffffu, a.v, o), __shfl_xor_sync(0xffffffffu, a.i, o)};
        a = better(a, t);
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) { redv[w] = a.v; redi[w] = a.i; }
    __syncthreads();
    ArgMax r{-INFINITY, 0x7fffffff};
    if (l < nw) r = ArgMax{redv[l], redi[l]};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        ArgMax t{__shfl_xor_sync(0xffffffffu, r.v, o), __shfl_xor_sync(0xffffffffu, r.i, o)};
        r = better(r, t);
    }
    return r;
}

__device__ int block_min_int(int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    int t = (l < nw) ? red[l] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = min(t, __shfl_xor_sync(0xffffffffu, t, o));
    return t;
}

__device__ int block_max_int(int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31, nw = blockDim.x >> 5;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    int t = (l < nw) ? red[l] : -1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    return t;
}

// Inclusive prefix sum over values held as VPT consecutive ids per thread.
template <int VPT>
__device__ void block_scan(float (&v)[VPT], float* red, float& total) {
    float run = 0.f;
#pragma unroll
    for (int j = 0; j < VPT; ++j) { run += v[j]; v[j] = run; }
    const int l = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    float x = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (l >= o) x += y;
    }
    __syncthreads();
    if (l == 31) red[w] = x;
    __syncthreads();
    if (w == 0) {
        float z = (l < nw) ? red[l] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, z, o);
            if (l >= o) z += y;
        }
        if (l < nw) red[l] = z;
    }
    __syncthreads();
    const float before = (x - run) + (w > 0 ? red[w - 1] : 0.f);
#pragma unroll
    for (int j = 0; j < VPT; ++j) v[j] += before;
    total = red[nw - 1];
}

// Inverse CDF over r (ids tid*VPT + j): smallest id with cumsum > u * sum; if rounding
// leaves none, the last id with positive mass.
template <int VPT>
__device__ int inverse_cdf(float (&r)[VPT], float u, float tau, bool& tie, float* redf, int* redi) {
    float cum[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) cum[j] = r[j];
    float total;
    block_scan<VPT>(cum, redf, total);
    const float thr = u * total;
    int first = 0x7fffffff, lastpos = -1;
    bool near = false;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int id = threadIdx.x * VPT + j;
        if (cum[j] > thr && id < first) first = id;
        if (r[j] > 0.f) lastpos = id;
        if (tau > 0.f && fabsf(cum[j] - thr) < tau * total) near = true;
    }
    first = block_min_int(first, redi);
    lastpos = block_max_int(lastpos, redi);
    const int nearany = block_max_int(near ? 1 : 0, redi);
    tie = tie || nearany;
    return (first != 0x7fffffff) ? first : lastpos;
}

// p = softmax(row * inv_temp) over ids tid*VPT + t, normalised; l keeps the raw logits and
// sq their per-thread sum of squares.
template <int VPT>
__device__ void softmax_row(const float* __restrict__ row, float inv_temp, float (&l)[VPT], float (&pr)[VPT],
                            float& sq, float* redf) {
    float mx = -INFINITY;
    sq = 0.f;
#pragma unroll
    for (int t = 0; t < VPT; ++t) {
        l[t] = row[threadIdx.x * VPT + t];
        mx = fmaxf(mx, l[t] * inv_temp);
        sq += l[t] * l[t];
    }
    mx = block_max(mx, redf);
    float se = 0.f;
#pragma unroll
    for (int t = 0; t < VPT; ++t) { pr[t] = __expf(l[t] * inv_temp - mx); se += pr[t]; }
    se = block_sum(se, redf);
    const float inv_se = 1.f / se;
#pragma unroll
    for (int t = 0; t < VPT; ++t) pr[t] *= inv_se;
}

// Several candidate blocks of sequence b under sampling, losslessly: rejection sampling
// applied recursively across the candidates that share the accepted path (a token tree with
// equal prefixes merged). At depth j the alive candidates are tried in index order against
// r (the lowest alive candidate's p at position j, then renormalised residuals
// max(0, r - q_c) after each rejection); an accepted draft x keeps alive the candidates whose
// draft j+1 is x. If all are rejected the correction is the inverse-CDF draw from r, after
// gamma acceptances the bonus from p at the path's end, both at u[lead][gamma]; the lowest
// alive candidate is committed. cand_k holds each candidate's drafts on the path, cand_corr
// the correction for the committed candidate and -1 for the others.
template <int VPT>
__device__ void accept_recursive(int b, const float* __restrict__ logits, int V, int C, int Tb, int gamma,
                                 float inv_temp, float tau, const int32_t* __restrict__ tokens,
                                 const float* __restrict__ qprob, const float* __restrict__ unif,
                                 int32_t* __restrict__ cand_k, int32_t* __restrict__ cand_corr,
                                 uint32_t* __restrict__ cand_tie, int32_t* __restrict__ out_k,
                                 int32_t* __restrict__ out_corr, int32_t* __restrict__ out_cand,
                                 uint32_t* __restrict__ out_tie, uint32_t* __restrict__ flags, float* redf,
                                 int* redi, float* pd_sh) {
    const int tid = threadIdx.x;
    auto draft = [&](int c, int j) {   // draft j+1 of candidate c, clamped like the embedding
        const int t = tokens[((size_t)b * C + c) * Tb + j + 1];
        return t < 0 ? 0 : (t >= V ? V - 1 : t);
    };
    uint32_t alive = C >= 32 ? 0xffffffffu : ((1u << C) - 1u);
    int k = gamma, corr = 0, lead = 0;
    bool tie = false;
    for (int j = 0; j <= gamma; ++j) {
        lead = __ffs(alive) - 1;
        float l[VPT], pr[VPT], sq;
        softmax_row<VPT>(logits + (((size_t)b * C + lead) * Tb + j) * V, inv_temp, l, pr, sq, redf);
        int x_acc = -1;
        for (int c = lead; j < gamma && c < C; ++c) {
            if (!((alive >> c) & 1u)) continue;
            const size_t bc = (size_t)b * C + c;
            const int x = draft(c, j);
            const float* qrow = qprob + (bc * gamma + j) * V;
            if (x / VPT == tid) {
#pragma unroll
                for (int t = 0; t < VPT; ++t)
                    if (tid * VPT + t == x) *pd_sh = pr[t];
            }
            __syncthreads();
            const float pd = *pd_sh;
            __syncthreads();
            const float lhs = unif[bc * Tb + j] * qrow[x];
            if (tau > 0.f && fabsf(lhs - pd) < tau * pd) tie = true;
            if (lhs < pd) {
                x_acc = x;
                break;
            }
            float r[VPT], rs = 0.f;
#pragma unroll
            for (int t = 0; t < VPT; ++t) {
                r[t] = fmaxf(pr[t] - qrow[tid * VPT + t], 0.f);
                rs += r[t];
            }
            rs = block_sum(rs, redf);
            if (rs > 0.f) {
                const float inv = 1.f / rs;
#pragma unroll
                for (int t = 0; t < VPT; ++t) pr[t] = r[t] * inv;
            } else if (tid == 0) {
                atomicOr(flags, (uint32_t)EVS_FLAG_EMPTY_RESIDUAL);
            }
        }
        if (x_acc < 0) {
            k = j;
            corr = inverse_cdf<VPT>(pr, unif[((size_t)b * C + lead) * Tb + gamma], tau, tie, redf, redi);
            break;
        }
        uint32_t keep = 0;
        for (int c = lead; c < C; ++c)
            if (((alive >> c) & 1u) && draft(c, j) == x_acc) keep |= 1u << c;
        if (tid == 0)
            for (int c = 0; c < C; ++c)
                if (((alive & ~keep) >> c) & 1u) cand_k[(size_t)b * C + c] = j;
        alive = keep;
    }
    if (tid == 0) {
        for (int c = 0; c < C; ++c) {
            const size_t bc = (size_t)b * C + c;
            if ((alive >> c) & 1u) cand_k[bc] = k;
            cand_corr[bc] = c == lead ? corr : -1;
            cand_tie[bc] = tie ? 1u : 0u;
        }
        out_k[b] = k;
        out_corr[b] = corr;
        if (out_cand) out_cand[b] = lead;
        if (out_tie) out_tie[b] = tie ? 1u : 0u;
    }
}

template <int VPT>
__global__ void __launch_bounds__(ACC_THREADS) accept_kernel(
    const float* __restrict__ logits, int V, int C, int Tb, int gamma, int mode, int rule, float inv_temp,
    float tau, const int32_t* __restrict__ tokens, const float* __restrict__ qprob,
    const float* __restrict__ unif, int32_t* __restrict__ cand_k, int32_t* __restrict__ cand_corr,
    uint32_t* __restrict__ cand_tie, int32_t* __restrict__ out_k, int32_t* __restrict__ out_corr,
    int32_t* __restrict__ out_cand, uint32_t* __restrict__ out_tie, uint32_t* __restrict__ flags) {
    pdl_trigger();
    pdl_wait();
    __shared__ float redf[32];
    __shared__ int redi[32];
    __shared__ float redv[32];
    __shared__ float pd_sh;
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    if (mode == EVS_MODE_SAMPLING && C > 1 && rule == EVS_CAND_RECURSIVE) {
        accept_recursive<VPT>(b, logits, V, C, Tb, gamma, inv_temp, tau, tokens, qprob, unif, cand_k, cand_corr,
                              cand_tie, out_k, out_corr, out_cand, out_tie, flags, redf, redi, &pd_sh);
        return;
    }
    int best_c = 0, best_k = -1, best_corr = 0;
    uint32_t any_tie = 0;
    for (int c = 0; c < C; ++c) {
        const int bc = b * C + c;
        int k = gamma, corr = 0;
        bool tie = false;
        for (int j = 0; j <= gamma; ++j) {
            const float* row = logits + ((size_t)bc * Tb + j) * V;
            float l[VPT], pr[VPT];
            float mx = -INFINITY, sq = 0.f;
#pragma unroll
            for (int t = 0; t < VPT; ++t) {
                l[t] = row[tid * VPT + t];
                mx = fmaxf(mx, l[t] * inv_temp);
                sq += l[t] * l[t];
            }
            mx = block_max(mx, redf);
            float se = 0.f;
#pragma unroll
            for (int t = 0; t < VPT; ++t) { pr[t] = __expf(l[t] * inv_temp - mx); se += pr[t]; }
            se = block_sum(se, redf);
            const float inv_se = 1.f / se;
#pragma unroll
            for (int t = 0; t < VPT; ++t) pr[t] *= inv_se;
            if (mode == EVS_MODE_GREEDY) {
                ArgMax a{-INFINITY, 0x7fffffff};
#pragma unroll
                for (int t = 0; t < VPT; ++t) a = better(a, ArgMax{l[t], tid * VPT + t});
                a = block_argmax(a, redv, redi);
                if (tau > 0.f) {
                    ArgMax s2{-INFINITY, 0x7fffffff};
#pragma unroll
                    for (int t = 0; t < VPT; ++t)
                        if (tid * VPT + t != a.i) s2 = better(s2, ArgMax{l[t], tid * VPT + t});
                    s2 = block_argmax(s2, redv, redi);
                    const float rms = sqrtf(block_sum(sq, redf) / (float)V);
                    if (a.v - s2.v < tau * rms) tie = true;
                }
                if (j < gamma && tokens[(size_t)bc * Tb + j + 1] == a.i) continue;
                k = j;
                corr = a.i;
                break;
            } else {
                const float u_last = unif[(size_t)bc * Tb + gamma];
                if (j < gamma) {
                    int dtok = tokens[(size_t)bc * Tb + j + 1];
                    dtok = dtok < 0 ? 0 : (dtok >= V ? V - 1 : dtok);
                    const float* qrow = qprob + ((size_t)bc * gamma + j) * V;
                    if (dtok / VPT == tid) {
#pragma unroll
                        for (int t = 0; t < VPT; ++t)
                            if (tid * VPT + t == dtok) pd_sh = pr[t];
                    }
                    __syncthreads();
                    const float pd = pd_sh;
                    __syncthreads();
                    const float lhs = unif[(size_t)bc * Tb + j] * qrow[dtok];
                    if (tau > 0.f && fabsf(lhs - pd) < tau * pd) tie = true;
                    if (lhs < pd) continue;
                    float r[VPT];
                    float rs = 0.f;
#pragma unroll
                    for (int t = 0; t < VPT; ++t) {
                        r[t] = fmaxf(pr[t] - qrow[tid * VPT + t], 0.f);
                        rs += r[t];
                    }
                    rs = block_sum(rs, redf);
                    if (!(rs > 0.f)) {
                        if (tid == 0) atomicOr(flags, (uint32_t)EVS_FLAG_EMPTY_RESIDUAL);
#pragma unroll
                        for (int t = 0; t < VPT; ++t) r[t] = pr[t];
                    }
                    k = j;
                    corr = inverse_cdf<VPT>(r, u_last, tau, tie, redf, redi);
                    break;
                }
                k = gamma;
                corr = inverse_cdf<VPT>(pr, u_last, tau, tie, redf, redi);
            }
        }
        if (tid == 0) {
            cand_k[bc] = k;
            cand_corr[bc] = corr;
            cand_tie[bc] = tie ? 1u : 0u;
        }
        if (k > best_k) { best_k = k; best_c = c; best_corr = corr; }
        any_tie |= tie ? 1u : 0u;
    }
    if (tid == 0) {
        out_k[b] = best_k;
        out_corr[b] = best_corr;
        if (out_cand) out_cand[b] = best_c;
        if (out_tie) out_tie[b] = any_tie;
    }
}

// =========================================================================================
// State slicing at k (Figure 1(d)): FIR tail <- stage rows k+1 .. k+L-1, IIR state <- s_k,
// and for several candidates the chosen candidate's k+1 block K/V rows into the cache;
// then kv_len = kv_base + k + 1. Grid (B, layers, blocks per layer): every layer runs in
// parallel, copies 16 bytes per thread where the rows allow it. s_k is not stored by the
// verify pass: it is k+1 steps of the diagonal recurrence from the pre-round state over the
// kept inputs, (k+1) d floats read instead of gamma+1 states of d N complex values written.
// =========================================================================================
template <typename T>
__global__ void slice_kernel(const LayerDesc* __restrict__ layers, int n_layers, int d, int dh,
                             int C, int Tb, int gamma, int t_max,
                             const int32_t* __restrict__ kin, const int32_t* __restrict__ cin,
                             const int32_t* __restrict__ kv_base, int32_t* __restrict__ kv_len,
                             uint32_t* __restrict__ flags) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x, li = blockIdx.y;
    const int k = kin[b];
    const int c = cin ? cin[b] : 0;
    const bool first = li == 0 && blockIdx.z == 0 && threadIdx.x == 0;
    if (k < 0 || k > gamma || c < 0 || c >= C) {
        if (first) atomicOr(flags, (uint32_t)EVS_FLAG_BAD_K);
        return;
    }
    const int bc = b * C + c;
    const int n0 = kv_base[b];
    const bool overflow = n0 + k + 1 > t_max;
    const int stride = gridDim.z * blockDim.x;
    const int start = blockIdx.z * blockDim.x + threadIdx.x;
    const LayerDesc L = layers[li];
    if (L.kind == EVS_LAYER_FIR) {
        const int Lm1 = L.param - 1;
        const float4* src = reinterpret_cast<const float4*>(L.stage + ((size_t)bc * (Lm1 + Tb) + k + 1) * d);
        float4* dst = reinterpret_cast<float4*>(L.tail + (size_t)b * Lm1 * d);
        for (int e = start; e < Lm1 * d / 4; e += stride) dst[e] = src[e];   // d % 64 == 0
    } else if (L.kind == EVS_LAYER_IIR) {
        // s_k from the pre-round state and the kept inputs u_0..u_k, by the scan's own
        // operations in the scan's order: the value the scan reached at position k. An item
        // is up to four poles of one channel, so each input load serves four recurrences.
        const int N = L.param, ppt = N < 4 ? N : 4, qpc = N / ppt;
        const float* u = L.uin + (size_t)bc * Tb * d;
        float2* st = L.state + (size_t)b * d * N;
        for (int it = start; it < d * qpc; it += stride) {
            const int ch = it / qpc;
            const size_t base = (size_t)ch * N + (size_t)(it % qpc) * ppt;
            float2 l[4], bq[4], s[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (q < ppt) {
                    l[q] = L.lam[base + q];
                    bq[q] = L.bq[base + q];
                    s[q] = st[base + q];
                }
            }
            for (int j0 = 0; j0 <= k; j0 += 8) {
                float uv[8];   // eight inputs requested before the recurrence uses any
#pragma unroll
                for (int j = 0; j < 8; ++j) uv[j] = j0 + j <= k ? u[(size_t)(j0 + j) * d + ch] : 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j0 + j <= k) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < ppt)
                                s[q] = make_float2(fmaf(l[q].x, s[q].x, fmaf(-l[q].y, s[q].y, bq[q].x * uv[j])),
                                                   fmaf(l[q].x, s[q].y, fmaf(l[q].y, s[q].x, bq[q].y * uv[j])));
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (q < ppt) st[base + q] = s[q];
        }
    } else if (C > 1 && !overflow) {
        const int H = L.param;
        const int per = (k + 1) * dh;
        for (int e = start; e < H * per; e += stride) {
            const int hh = e / per, r = e % per;
            const int j = r / dh, x = r % dh;
            const size_t srci = ((((size_t)bc) * H + hh) * Tb + j) * dh + x;
            const size_t dsti = (((size_t)b * H + hh) * t_max + n0 + j) * dh + x;
            ((T*)L.kc)[dsti] = ((const T*)L.ks)[srci];
            ((T*)L.vc)[dsti] = ((const T*)L.vs)[srci];
        }
    }
    if (first) {
        if (overflow) atomicOr(flags, (uint32_t)EVS_FLAG_KV_OVERFLOW);
        kv_len[b] = overflow ? t_max : n0 + k + 1;
    }
}

__global__ void advance_kernel(const int32_t* __restrict__ kv_base, int32_t* __restrict__ kv_len,
                               int B, int T, int t_max, uint32_t* __restrict__ flags) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int nl = kv_base[b] + T;
    if (nl > t_max) { atomicOr(flags, (uint32_t)EVS_FLAG_KV_OVERFLOW); nl = t_max; }
    kv_len[b] = nl;
}

// =========================================================================================
// launchers
// =========================================================================================
static inline bool is_bf16(const evs_handle* h) { return h->cfg.dtype == EVS_DTYPE_BF16; }
using bf16 = __nv_bfloat16;

void launch_embed(evs_handle* h, const int32_t* tokens, int tok_stride_bc, const int32_t* anchor,
                  const Pass& p) {
    prof_begin(h, EVS_K_EMBED);
    const int d = h->cfg.d;
    if (is_bf16(h))
        launch_k(h, embed_kernel<bf16>, dim3(p.M), dim3(256), 0, (const bf16*)h->w.embed, tokens, tok_stride_bc,
            anchor, h->h, d, p.C, p.T, h->cfg.vocab, p.B, h->kv_len, h->kv_base, h->flags,
            h->fused ? h->hb : nullptr, h->fused ? h->ssq : nullptr, d / 128, h->g.M_max);
    else
        launch_k(h, embed_kernel<float>, dim3(p.M), dim3(256), 0, (const float*)h->w.embed, tokens, tok_stride_bc,
            anchor, h->h, d, p.C, p.T, h->cfg.vocab, p.B, h->kv_len, h->kv_base, h->flags,
            (__nv_bfloat16*)nullptr, (float*)nullptr, 0, 0);
    h->launches++;
    prof_end(h, EVS_K_EMBED);
}

void launch_rmsnorm(evs_handle* h, const Pass& p) {
    prof_begin(h, EVS_K_NORM);
    const int d = h->cfg.d;
    if (is_bf16(h)) launch_k(h, rmsnorm_kernel<bf16>, dim3(p.M), dim3(256), 0, h->h, (bf16*)h->act, d);
    else launch_k(h, rmsnorm_kernel<float>, dim3(p.M), dim3(256), 0, h->h, (float*)h->act, d);
    h->launches++;
    prof_end(h, EVS_K_NORM);
}

void launch_gemm(evs_handle* h, const void* A, const void* W, float* Y, int M, int N, int K, int ldy,
                 int accumulate, const GemmFuse* fz, int* fused) {
    prof_begin(h, EVS_K_GEMM);
    if (fused) *fused = 0;
    if (is_bf16(h) && gemm_tc_supported(M, N, K) &&
        launch_gemm_tc(h, A, h->g.M_max, W, Y, M, N, K, ldy, accumulate, fz, fused)) {
        h->launches++;
        prof_end(h, EVS_K_GEMM);
        return;
    }
    dim3 grid((N + GS_BN - 1) / GS_BN, (M + GS_BM - 1) / GS_BM);
    if (is_bf16(h))
        launch_k(h, gemm_simt_kernel<bf16>, dim3(grid), dim3(256), 0, (const bf16*)A, (const bf16*)W, Y, M, N, K, ldy,
                                                             accumulate);
    else
        launch_k(h, gemm_simt_kernel<float>, dim3(grid), dim3(256), 0, (const float*)A, (const float*)W, Y, M, N, K,
                                                              ldy, accumulate);
    h->launches++;
    prof_end(h, EVS_K_GEMM);
}

void launch_fir(evs_handle* h, int li, const Pass& p) {
    prof_begin(h, EVS_K_FIR);
    const int d = h->cfg.d;
    const LayerDesc& L = h->layer[li];
    const float* taps = h->w.layer[li].fir_taps;
    dim3 grid((d + 63) / 64, p.B * p.C);
    if (is_bf16(h))
        launch_k(h, fir_kernel<bf16>, dim3(grid), dim3(64), 0, h->y, 3 * d, (bf16*)h->act, d, p.C, p.T, p.commit, taps,
                                                       L.param, L.tail, L.stage);
    else
        launch_k(h, fir_kernel<float>, dim3(grid), dim3(64), 0, h->y, 3 * d, (float*)h->act, d, p.C, p.T, p.commit,
                                                        taps, L.param, L.tail, L.stage);
    h->launches++;
    prof_end(h, EVS_K_FIR);
}

void launch_iir(evs_handle* h, int li, const Pass& p, const float* u, int ldu) {
    prof_begin(h, EVS_K_IIR);
    const int d = h->cfg.d;
    const LayerDesc& L = h->layer[li];
    const int N = L.param;
    dim3 grid((d * N + 255) / 256, p.B * p.C);
    const float2* lam = (const float2*)h->w.layer[li].iir_lambda;
    const float2* bb = (const float2*)h->w.layer[li].iir_b;
    const float2* cc = (const float2*)h->w.layer[li].iir_c;
#define EVS_IIR(TY, NP)                                                                                       \
    launch_k(h, iir_kernel<TY, NP>, dim3(grid), dim3(256), 0, u, ldu, (TY*)h->act, d, N, p.C, p.T, p.commit, lam, \
             bb, cc, L.state)
#define EVS_IIRC(TY, NP)                                                                                      \
    launch_k(h, iir_quad_kernel<TY, NP>, dim3((d * (NP < 4 ? 1 : NP / 4) + 255) / 256, p.B * p.C), dim3(256), 0,     \
             u, ldu, (TY*)h->act, d, p.C, p.T, p.commit, lam, bb, cc, L.state)
    const int lpc = N < 4 ? 1 : N / 4;
    if ((d * lpc) % 32 != 0) {   // the quad kernel's early exit must take whole warps
        if (is_bf16(h)) EVS_IIR(bf16, 0); else EVS_IIR(float, 0);
    } else if (is_bf16(h)) {
        switch (N) {
            case 1: EVS_IIRC(bf16, 1); break;
            case 2: EVS_IIRC(bf16, 2); break;
            case 4: EVS_IIRC(bf16, 4); break;
            case 8: EVS_IIRC(bf16, 8); break;
            case 16: EVS_IIRC(bf16, 16); break;
            default: EVS_IIR(bf16, 0); break;
        }
    } else {
        switch (N) {
            case 1: EVS_IIRC(float, 1); break;
            case 2: EVS_IIRC(float, 2); break;
            case 4: EVS_IIRC(float, 4); break;
            case 8: EVS_IIRC(float, 8); break;
            case 16: EVS_IIRC(float, 16); break;
            default: EVS_IIR(float, 0); break;
        }
    }
#undef EVS_IIRC
#undef EVS_IIR
    h->launches++;
    prof_end(h, EVS_K_IIR);
}

void launch_kv_write(evs_handle* h, int li, const Pass& p) {
    prof_begin(h, EVS_K_KV_WRITE);
    const int d = h->cfg.d;
    const LayerDesc& L = h->layer[li];
    const int H = L.param, dh = h->cfg.head_dim;
    dim3 grid((d + 255) / 256, p.M);
    if (is_bf16(h))
        launch_k(h, kv_write_kernel<bf16>, dim3(grid), dim3(256), 0, h->y, 3 * d, d, H, dh, p.C, p.T, p.kv_in_cache,
            h->cfg.t_max, h->kv_base, (bf16*)L.kc, (bf16*)L.vc, (bf16*)L.ks, (bf16*)L.vs, h->flags);
    else
        launch_k(h, kv_write_kernel<float>, dim3(grid), dim3(256), 0, h->y, 3 * d, d, H, dh, p.C, p.T, p.kv_in_cache,
            h->cfg.t_max, h->kv_base, (float*)L.kc, (float*)L.vc, (float*)L.ks, (float*)L.vs, h->flags);
    h->launches++;
    prof_end(h, EVS_K_KV_WRITE);
}

void launch_attention(evs_handle* h, int li, const Pass& p) {
    prof_begin(h, EVS_K_ATTN);
    const int d = h->cfg.d;
    const LayerDesc& L = h->layer[li];
    const int H = L.param, dh = h->cfg.head_dim;
    const int Q = p.C * p.T;
    const Geometry& g = h->g;
    const AttnPlan& plan = p.commit ? h->plan_prefill : h->plan_verify;
    int splits = g.kv_splits, chunk = g.kv_chunk, fa_grid = 0;
    if (plan.ok && launch_attn_tensor(h, li, p, plan)) {
        splits = plan.splits;
        chunk = 0;                               // every slot written (empty ones m = -inf)
        fa_grid = plan.runs ? kAttnGrid : 0;     // or runs of key tiles over the persistent grid
    } else {
    dim3 grid(g.kv_splits, p.B * H, (Q + AQ - 1) / AQ);
    if (is_bf16(h))
        launch_k(h, attn_split_kernel<bf16>, dim3(grid), dim3(256), 0, h->y, 3 * d, (const bf16*)L.kc, (const bf16*)L.vc,
            H, dh, Q, g.q_max, h->cfg.t_max, g.kv_chunk, g.kv_splits, h->kv_base, h->attn_part);
    else
        launch_k(h, attn_split_kernel<float>, dim3(grid), dim3(256), 0, h->y, 3 * d, (const float*)L.kc,
            (const float*)L.vc, H, dh, Q, g.q_max, h->cfg.t_max, g.kv_chunk, g.kv_splits, h->kv_base,
            h->attn_part);
    }
    h->launches++;
    prof_end(h, EVS_K_ATTN);
    prof_begin(h, EVS_K_ATTN_COMBINE);
    dim3 grid2(p.B * H, p.C, (p.T + 3) / 4);
    // more CTAs than one wave at four an SM: the smaller batch, for a fifth CTA an SM
    const bool waves = (long long)grid2.x * grid2.y * grid2.z > 4LL * kAttnGrid;
#define EVS_CMB(TY, EPL)                                                                                    \
    do {                                                                                                    \
        if (waves)                                                                                          \
            launch_k(h, attn_combine_kernel<TY, EPL, 4>, dim3(grid2), dim3(128), 0, h->y, 3 * d,            \
                     (const TY*)L.kc, (const TY*)L.vc, (const TY*)L.ks, (const TY*)L.vs, H, dh, p.C, p.T, Q, \
                     g.q_max, h->cfg.t_max, splits, chunk, p.B, fa_grid, p.kv_in_cache, h->kv_base,        \
                     h->attn_part, (TY*)h->act, d);                                                         \
        else                                                                                                \
            launch_k(h, attn_combine_kernel<TY, EPL, 8>, dim3(grid2), dim3(128), 0, h->y, 3 * d,            \
                     (const TY*)L.kc, (const TY*)L.vc, (const TY*)L.ks, (const TY*)L.vs, H, dh, p.C, p.T, Q, \
                     g.q_max, h->cfg.t_max, splits, chunk, p.B, fa_grid, p.kv_in_cache, h->kv_base,        \
                     h->attn_part, (TY*)h->act, d);                                                         \
    } while (0)
    if (is_bf16(h)) {
        if (dh > 64) EVS_CMB(bf16, 4); else if (dh > 32) EVS_CMB(bf16, 2); else EVS_CMB(bf16, 1);
    } else {
        if (dh > 64) EVS_CMB(float, 4); else if (dh > 32) EVS_CMB(float, 2); else EVS_CMB(float, 1);
    }
#undef EVS_CMB
    h->launches++;
    prof_end(h, EVS_K_ATTN_COMBINE);
}

void launch_accept(evs_handle* h, const int32_t* tokens, const float* q, const float* u, int32_t* acc,
                   int32_t* corr, int32_t* cand, uint32_t* tie) {
    prof_begin(h, EVS_K_ACCEPT);
    const evs_config& c = h->cfg;
    const int V = c.vocab;
    const float inv_t = 1.0f / c.temperature;
    const int Tb = c.gamma + 1;
#define EVS_ACC(VPT)                                                                              \
    launch_k(h, accept_kernel<VPT>, dim3(c.batch), dim3(ACC_THREADS), 0, h->logits, V, c.n_cand, Tb, c.gamma,   \
        c.mode, c.cand_rule, inv_t, c.near_tie_tau, tokens, q, u, h->cand_k, h->cand_corr, h->cand_tie, acc, \
        corr, cand, tie, h->flags)
    switch (V / ACC_THREADS) {
        case 1: EVS_ACC(1); break;
        case 2: EVS_ACC(2); break;
        case 4: EVS_ACC(4); break;
        case 8: EVS_ACC(8); break;
        default: EVS_ACC(16); break;
    }
#undef EVS_ACC
    h->launches++;
    prof_end(h, EVS_K_ACCEPT);
}

// The next-token draw of a decode step: the acceptance kernel over one candidate of one
// position with no drafts (gamma 0), so it returns the argmax or the inverse-CDF draw at
// u[b] of the position's distribution. The per-candidate words and k (always 0) land in
// the handle's candidate scratch.
void launch_pick(evs_handle* h, const float* u, int32_t* next, uint32_t* tie) {
    prof_begin(h, EVS_K_ACCEPT);
    const evs_config& c = h->cfg;
    const int V = c.vocab;
    const float inv_t = 1.0f / c.temperature;
#define EVS_PICK(VPT)                                                                             \
    launch_k(h, accept_kernel<VPT>, dim3(c.batch), dim3(ACC_THREADS), 0, h->logits, V, 1, 1, 0, c.mode, 0, inv_t, \
        c.near_tie_tau, (const int32_t*)nullptr, (const float*)nullptr, u, h->cand_k, h->cand_corr,            \
        h->cand_tie, h->cand_k, next, (int32_t*)nullptr, tie, h->flags)
    switch (V / ACC_THREADS) {
        case 1: EVS_PICK(1); break;
        case 2: EVS_PICK(2); break;
        case 4: EVS_PICK(4); break;
        case 8: EVS_PICK(8); break;
        default: EVS_PICK(16); break;
    }
#undef EVS_PICK
    h->launches++;
    prof_end(h, EVS_K_ACCEPT);
}

void launch_slice(evs_handle* h, const int32_t* k, const int32_t* cand) {
    prof_begin(h, EVS_K_SLICE);
    const evs_config& c = h->cfg;
    // blocks per layer: enough for one item per thread on the largest layer (an IIR layer's
    // channels x pole quads, a FIR tail in float4, a candidate's K/V rows), 8 to 64
    long long items = 0;
    for (int i = 0; i < c.n_layers; ++i) {
        const int kind = c.layer_kind[i], prm = c.layer_param[i];
        if (kind == EVS_LAYER_IIR) items = std::max(items, (long long)c.d * std::max(prm / 4, 1));
        else if (kind == EVS_LAYER_FIR) items = std::max(items, (long long)(prm - 1) * c.d / 4);
        else if (c.n_cand > 1) items = std::max(items, (long long)c.d * (c.gamma + 1));
    }
    dim3 grid(c.batch, c.n_layers, (unsigned)std::min(64LL, std::max(8LL, (items + 255) / 256)));
    if (is_bf16(h))
        launch_k(h, slice_kernel<bf16>, dim3(grid), dim3(256), 0, h->layer_dev, c.n_layers, c.d, c.head_dim, c.n_cand,
            c.gamma + 1, c.gamma, c.t_max, k, cand, h->kv_base, h->kv_len, h->flags);
    else
        launch_k(h, slice_kernel<float>, dim3(grid), dim3(256), 0, h->layer_dev, c.n_layers, c.d, c.head_dim, c.n_cand,
            c.gamma + 1, c.gamma, c.t_max, k, cand, h->kv_base, h->kv_len, h->flags);
    h->launches++;
    prof_end(h, EVS_K_SLICE);
}

void launch_advance(evs_handle* h, int T) {
    prof_begin(h, EVS_K_ADVANCE);
    launch_k(h, advance_kernel, dim3(1), dim3(256), 0, h->kv_base, h->kv_len, h->cfg.batch, T, h->cfg.t_max, h->flags);
    h->launches++;
    prof_end(h, EVS_K_ADVANCE);
}

}  // namespace evs
