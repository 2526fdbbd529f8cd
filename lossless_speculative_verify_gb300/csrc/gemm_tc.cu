// Weight-streaming skinny projection on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA. Y[m][n] (+)= sum_k X[m][k] W[n][k] with X the block's activations (M =
// sequences x candidates x (gamma+1) rows, a few to a few hundred) and W an out-major
// weight matrix streamed from HBM exactly once per launch.
//
// Swap-AB: the weight tile is the 128-row A operand and the tokens are the N dimension of
// the MMA (16..256 per instruction, up to 512 in two accumulators), so the accumulator
// D[n][m] sits in TMEM with one output channel per lane. One CTA owns a 128-channel tile
// and a range of K; ranges of K are split across CTAs until the grid fills the 152 SMs,
// and the last CTA to finish a tile adds the partial sums in a fixed order (deterministic).
//
// Roles in a CTA of 128 threads: thread 0 issues TMA loads into a ring of stages, thread
// 32 issues the MMAs and releases stages with tcgen05.commit, then all four warps read
// their 32 TMEM lanes for the epilogue.
#include <cudaTypedefs.h>

#include "evs_common.cuh"
#include "sm100_ptx.cuh"

namespace evs {

constexpr int TC_BM = 128;                    // output channels per tile (MMA M)
constexpr int TC_BK = 64;                     // K per stage: one 128-byte swizzled row of bf16
constexpr int TC_A_BYTES = TC_BM * TC_BK * 2; // 16 KiB
constexpr int TC_SMEM_BUDGET = 200 * 1024;

struct TcArgs {
    float* Y;
    int ldy, M, N, kblocks, splits, n_pad, stages, accumulate, ncols;
    float* part;      // [splits][M][N] partial sums when splits > 1
    int* counters;    // [N / 128] arrival counters, zero between launches
    uint32_t* flags;
};

__global__ void __launch_bounds__(128, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot[1];
    __shared__ volatile int abort_flag[1];
    __shared__ int last_flag[1];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const int b_bytes = p.n_pad * 128;
    uint8_t* sA = smem;
    uint8_t* sB = smem + (size_t)p.stages * TC_A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + (size_t)p.stages * b_bytes);
    uint64_t* empty = full + p.stages;
    uint64_t* done = empty + p.stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int n0 = tile * TC_BM;
    const int kb0 = (int)((long long)p.kblocks * split / p.splits);
    const int kb1 = (int)((long long)p.kblocks * (split + 1) / p.splits);
    const int nk = kb1 - kb0;

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
        for (int i = 0; i < nk; ++i) {
            const int s = i % p.stages;
            const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
            if (i >= p.stages && !mbar_wait(&empty[s], ph ^ 1u)) { *abort_flag = 1; break; }
            mbar_arrive_expect_tx(&full[s], (uint32_t)(TC_A_BYTES + b_bytes));
            const int k = (kb0 + i) * TC_BK;
            tma_load_2d(sA + (size_t)s * TC_A_BYTES, &tmA, k, n0, &full[s], pol_w);
            for (int r = 0; r < p.n_pad; r += 256)
                tma_load_2d(sB + (size_t)s * b_bytes + (size_t)r * 128, &tmB, k, r, &full[s], pol_x);
        }
    } else if (threadIdx.x == 32) {
        // ---- MMA issuer ------------------------------------------------------------------
        const int n_hi = p.n_pad > 256 ? p.n_pad - 256 : 0;
        const int n_lo = p.n_pad - n_hi;
        const uint32_t id_lo = idesc_bf16_f32(TC_BM, n_lo);
        const uint32_t id_hi = idesc_bf16_f32(TC_BM, n_hi > 0 ? n_hi : 16);
        for (int i = 0; i < nk; ++i) {
            const int s = i % p.stages;
            const uint32_t ph = (uint32_t)(i / p.stages) & 1u;
            if (!mbar_wait(&full[s], ph)) { *abort_flag = 1; break; }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + (size_t)s * TC_A_BYTES);
            const uint32_t b0 = smem_u32(sB + (size_t)s * b_bytes);
#pragma unroll
            for (int kk = 0; kk < TC_BK / 16; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + kk * 32);
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16(tmem, ad, smem_desc_sw128(b0 + kk * 32), id_lo, acc);
                if (n_hi > 0) tc_mma_f16(tmem + 256, ad, smem_desc_sw128(b0 + 256 * 128 + kk * 32), id_hi, acc);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(done);
    }

    // ---- epilogue: lane = output channel, columns = tokens ---------------------------------
    __syncwarp();
    const bool ok = mbar_wait(done, 0);
    tc_fence_after();
    const bool bad = !ok || *abort_flag;
    if (bad && threadIdx.x == 0) atomicOr(p.flags, (uint32_t)EVS_FLAG_TIMEOUT);
    const int n = n0 + warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const bool col_ok = n < p.N && !bad;
    if (p.splits == 1) {
        for (int c0 = 0; c0 < p.M; c0 += 16) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = c0 + j;
                if (m < p.M && col_ok) {
                    float* dst = p.Y + (size_t)m * p.ldy + n;
                    *dst = p.accumulate ? (*dst + v[j]) : v[j];
                }
            }
        }
    } else {
        float* mine = p.part + (size_t)split * p.M * p.N;
        for (int c0 = 0; c0 < p.M; c0 += 16) {
            float v[16];
            tmem_ld16(trow + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int m = c0 + j;
                if (m < p.M && col_ok) mine[(size_t)m * p.N + n] = v[j];
            }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) *last_flag = (atomicAdd(&p.counters[tile], 1) == p.splits - 1);
        __syncthreads();
        if (*last_flag) {
            __threadfence();
            if (col_ok) {
                for (int m = 0; m < p.M; ++m) {
                    float s = 0.f;
                    for (int sp = 0; sp < p.splits; ++sp) s += __ldcg(p.part + ((size_t)sp * p.M + m) * p.N + n);
                    float* dst = p.Y + (size_t)m * p.ldy + n;
                    *dst = p.accumulate ? (*dst + s) : s;
                }
            }
            if (threadIdx.x == 0) p.counters[tile] = 0;
        }
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
int gemm_tc_init() {
    int dev = 0, optin = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, gemm_tc_kernel) != cudaSuccess)
        return -1;
    const int dyn = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn) != cudaSuccess)
        return -1;
    return dyn;
}

// Split K only as far as each CTA still streams at least 8 k-blocks (128 KiB of weights),
// and no further than filling the 152 SMs once: past that the partial-sum round trip and
// the per-CTA start-up cost more than the extra parallelism returns.
int tc_splits(int N, int K) {
    const int tiles = N / TC_BM, kblocks = K / TC_BK;
    int s = 152 / tiles;
    if (s > kblocks / 8) s = kblocks / 8;
    if (s < 1) s = 1;
    return s;
}

bool gemm_tc_supported(int M, int N, int K) {
    return M >= 1 && M <= 512 && N % TC_BM == 0 && K % TC_BK == 0 && N > 0 && K > 0;
}

// Returns false (nothing launched) if a tensor map could not be built.
bool launch_gemm_tc(evs_handle* h, const void* X, int x_rows, const void* W, float* Y, int M, int N, int K,
                    int ldy, int accumulate) {
    // tokens padded to the MMA's N granularity; above 256 two accumulators of 256 columns
    const int n_pad = M > 256 ? 512 : (M + 15) / 16 * 16;
    CUtensorMap ta, tb;
    if (!make_map(&ta, W, (uint64_t)N, (uint64_t)K, TC_BM)) return false;
    if (!make_map(&tb, X, (uint64_t)x_rows, (uint64_t)K, (uint32_t)(n_pad < 256 ? n_pad : 256))) return false;
    const int tiles = N / TC_BM, kblocks = K / TC_BK;
    const int splits = tc_splits(N, K);
    const int per = (kblocks + splits - 1) / splits;
    const int stage_bytes = TC_A_BYTES + n_pad * 128;
    int stages = TC_SMEM_BUDGET / stage_bytes;
    if (stages > per) stages = per;
    if (stages < 1) stages = 1;
    int ncols = 32;
    while (ncols < n_pad) ncols <<= 1;
    const size_t smem = (size_t)stages * stage_bytes + 1024 + (2 * stages + 1) * 8;
    if ((int)smem > h->tc_smem_max) return false;
    TcArgs a{Y, ldy, M, N, kblocks, splits, n_pad, stages, accumulate, ncols, h->gemm_part, h->gemm_counters,
             h->flags};
    gemm_tc_kernel<<<dim3(tiles, splits), 128, smem, h->stream>>>(ta, tb, a);
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
// limit. Filled by the first call on each device.
NoAllocScratch* g_noalloc_ptr[kNoAllocMaxDevices];
int g_noalloc_smem[kNoAllocMaxDevices];

}  // namespace
}  // namespace evs

extern "C" evs_status evs_projection_noalloc(const void* X, int32_t x_rows, const void* W, float* Y, int32_t M,
                                             int32_t N, int32_t K, int32_t ldy, int32_t accumulate,
                                             void* stream) {
    using namespace evs;
    if (!X || !W || !Y || !gemm_tc_supported(M, N, K) || x_rows < M || ldy < N || N / TC_BM > kNoAllocCounters)
        return EVS_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return EVS_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return EVS_ERR_INVALID_ARG;
    if (!g_noalloc_ptr[dev]) {
        // one-time set-up on this device (the device is current here)
        NoAllocScratch* p = nullptr;
        if (cudaGetSymbolAddress((void**)&p, g_noalloc_scratch) != cudaSuccess || !p) return EVS_ERR_CUDA;
        const int smem_max = gemm_tc_init();
        if (smem_max < 0) return EVS_ERR_CUDA;
        g_noalloc_smem[dev] = smem_max;
        g_noalloc_ptr[dev] = p;
    }
    NoAllocScratch* sc = g_noalloc_ptr[dev];
    const int splits = tc_splits(N, K);
    if (splits > 1 && (size_t)splits * M * N > kNoAllocPartFloats) return EVS_ERR_CAPACITY;
    const int n_pad = M > 256 ? 512 : (M + 15) / 16 * 16;
    CUtensorMap ta, tb;
    if (!make_map(&ta, W, (uint64_t)N, (uint64_t)K, TC_BM)) return EVS_ERR_CUDA;
    if (!make_map(&tb, X, (uint64_t)x_rows, (uint64_t)K, (uint32_t)(n_pad < 256 ? n_pad : 256))) return EVS_ERR_CUDA;
    const int tiles = N / TC_BM, kblocks = K / TC_BK;
    const int per = (kblocks + splits - 1) / splits;
    const int stage_bytes = TC_A_BYTES + n_pad * 128;
    int stages = TC_SMEM_BUDGET / stage_bytes;
    if (stages > per) stages = per;
    if (stages < 1) stages = 1;
    int ncols = 32;
    while (ncols < n_pad) ncols <<= 1;
    const size_t smem = (size_t)stages * stage_bytes + 1024 + (2 * stages + 1) * 8;
    if ((int)smem > g_noalloc_smem[dev]) return EVS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    // the array keeps the previous call's contents: the counters must start at zero
    if (cudaMemsetAsync(sc->counters, 0, sizeof(sc->counters), s) != cudaSuccess) return EVS_ERR_CUDA;
    TcArgs a{Y, ldy, M, N, kblocks, splits, n_pad, stages, accumulate, ncols, sc->part, sc->counters, &sc->flags};
    gemm_tc_kernel<<<dim3(tiles, splits), 128, smem, s>>>(ta, tb, a);
    return cudaGetLastError() == cudaSuccess ? EVS_OK : EVS_ERR_CUDA;
}

