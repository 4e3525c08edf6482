// No-split-K bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA.  C[M, N] = A[M, K] * B[N, K]^T with fp32 accumulation.
//
// Batch invariance ([DVR] para 1: batch-invariant matmul never splits K and
// always uses the same data-parallel tiling): every output tile is owned by
// one CTA, whose single MMA thread walks K from 0 upwards in steps of 16
// (tcgen05.mma kind::f16, M = 128) into one TMEM accumulator.  The sequence of
// MMAs that produces C[m][n] -- which k-chunks, in which order, into one
// accumulator -- is the same for every M, every tile width and every row
// position inside the tile; the tensor core computes each output element of an
// MMA independently of the instruction's N (checked bitwise on the GPU for
// N = 16..256), so the tile width is free to follow the problem size.
//
// Kernel layout (192 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: A tile [a_rows x 64] and B tile [BN x 64] per
//               stage, 128-byte swizzle, mbarrier transaction counts.  For
//               M <= 128 only the real rows of A are copied (a_rows =
//               M rounded up to 8); the rest of each A stage is zeroed once.
//   warp 1      TMEM allocator + single-thread MMA issuer; commits free smem
//               stages and publish finished accumulators.
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 16 columns, convert, store.
// Two accumulators in TMEM let the epilogue of tile i overlap the MMAs of
// tile i + 1.  Up to 24 stages keep a whole small weight slice in flight.
// Launched with programmatic dependent launch: barrier set-up, TMEM
// allocation and the zero fill overlap the previous kernel.  Every wait is
// bounded (2 s); on time-out the kernel raises BIV_DEVERR_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_gemm_err)

constexpr int kBM = 128;
constexpr int kBK = 64;                       // 64 bf16 = one 128-byte swizzle row
constexpr int kABytes = kBM * kBK * 2;        // full A stage (16 KiB)
constexpr int kRingBudget = 200 * 1024;       // bytes of pipeline stages per CTA
constexpr int kMaxStages = 24;
constexpr int kBarBytes = 512;
constexpr int kWave = 152;                    // CTAs of one wave on a 152-SM part

struct GemmArgs {
    int M, N, K;
    int BN;          // tile width (multiple of 16, 16..256)
    int stages;      // ring depth
    int a_rows;      // rows of A copied per stage (multiple of 8, <= 128)
    uint32_t idesc;  // tcgen05 instruction descriptor for M=128, N=BN
    uint32_t tmem_cols;
};

inline int stage_bytes(int BN) { return kABytes + BN * kBK * 2; }

template <bool OUT_F32>
__global__ void __launch_bounds__(192, 1)
gemm_nosplitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     void* __restrict__ C, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int STAGE = kABytes + g.BN * kBK * 2;
    const int S = g.stages;
    uint8_t* tiles = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE);
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;     // [2]
    uint64_t* tempty = tfull + 2;             // [2]
    uint64_t* drain = tempty + 2;             // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = g.M, N = g.N, BN = g.BN;
    const int m_tiles = (M + kBM - 1) / kBM;
    const int n_tiles = (N + BN - 1) / BN;
    const int n_work = m_tiles * n_tiles;
    const int KB = (g.K + kBK - 1) / kBK;
    const uint32_t tx_bytes = static_cast<uint32_t>(g.a_rows * kBK * 2 + BN * kBK * 2);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 128);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, g.tmem_cols);
        tmem_relinquish();
    }
    // Rows of A that TMA does not write stay zero for the whole kernel.
    if (g.a_rows < kBM) {
        const int zero_off = g.a_rows * kBK * 2;
        const int chunks = (kABytes - zero_off) / 16;
        for (int s = 0; s < S; ++s) {
            uint4* z = reinterpret_cast<uint4*>(tiles + s * STAGE + zero_off);
            for (int i = threadIdx.x; i < chunks; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();       // inputs of the previous kernel are complete and visible from here on
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            const uint64_t pol_a = policy_evict_last();    // activations: reused by every CTA
            const uint64_t pol_b = policy_evict_first();   // weights: streamed once
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_work && ok; t += gridDim.x) {
                const int n_blk = t / m_tiles;
                const int m_blk = t - n_blk * m_tiles;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_gemm_err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = tiles + stage * STAGE;
                    mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    tma_load_2d(sa, &tmA, &full[stage], kb * kBK, m_blk * kBM, pol_a);
                    tma_load_2d(sa + kABytes, &tmB, &full[stage], kb * kBK, n_blk * BN, pol_b);
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the copies that may still be in flight land before the CTA exits.
                long long first = issued > S ? issued - S : 0;
                for (long long i = first; i < issued; ++i)
                    mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int t = blockIdx.x; t < n_work && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, &g_gemm_err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, &g_gemm_err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + stage * STAGE);
                    const uint64_t a_desc = sw128_kmajor_desc(a_addr);
                    const uint64_t b_desc = sw128_kmajor_desc(a_addr + kABytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        // +32 bytes along K inside the swizzle row = +2 in 16-byte units.
                        umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, g.idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    any = true;
                    umma_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                umma_commit(drain);               // all MMAs issued so far have finished
                mbar_wait_drain(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < n_work; t += gridDim.x) {
            const int n_blk = t / m_tiles;
            const int m_blk = t - n_blk * m_tiles;
            if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, &g_gemm_err)) break;
            tc_fence_after();
            const int row = m_blk * kBM + q * 32 + lane;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c), r);
                tmem_ld_wait();
                if (row < M) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = n_blk * BN + c + h * 8;
                        if (col < N) {
                            const uint32_t* v = r + h * 8;
                            if constexpr (OUT_F32) {
                                float4* dst = reinterpret_cast<float4*>(
                                    static_cast<float*>(C) + static_cast<long long>(row) * N + col);
                                dst[0] = make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]),
                                                     __uint_as_float(v[2]), __uint_as_float(v[3]));
                                dst[1] = make_float4(__uint_as_float(v[4]), __uint_as_float(v[5]),
                                                     __uint_as_float(v[6]), __uint_as_float(v[7]));
                            } else {
                                uint4 o;
                                o.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
                                o.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
                                o.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
                                o.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
                                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(C) +
                                                          static_cast<long long>(row) * N + col) = o;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, g.tmem_cols);
}

// --------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Row-major bf16 [rows, cols] viewed by TMA as boxes of [box_rows x 64], 128-B swizzle.
bool encode_kmajor(CUtensorMap* map, const void* base, int cols, int rows, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

uint32_t tmem_cols_for(int BN) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(2 * BN)) c <<= 1;
    return c;
}

template <bool F32>
int launch_gemm(const void* A, const void* B, void* C, int M, int N, int K, int BN, cudaStream_t stream) {
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.BN = BN;
    g.stages = std::min(kMaxStages, kRingBudget / stage_bytes(BN));
    g.a_rows = M >= kBM ? kBM : ((M + 7) / 8) * 8;
    g.idesc = idesc_bf16_f32(kBM, BN);
    g.tmem_cols = tmem_cols_for(BN);
    CUtensorMap ta, tb;
    if (!encode_kmajor(&ta, A, K, M, g.a_rows) || !encode_kmajor(&tb, B, K, N, BN)) {
        set_cuda_error(cudaErrorInvalidValue);
        return BIV_ERR_CUDA;
    }
    const int smem = 1024 + g.stages * stage_bytes(BN) + kBarBytes;
    auto kern = gemm_nosplitk_kernel<F32>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             1024 + kRingBudget + kBarBytes);
        if (e != cudaSuccess) return cuda_status(e);
        configured_device = dev;
    }
    const long long work = static_cast<long long>((M + kBM - 1) / kBM) * ((N + BN - 1) / BN);
    const int grid = static_cast<int>(std::min<long long>(work, num_sms()));
    return launch_pdl(kern, dim3(grid), dim3(192), static_cast<size_t>(smem), stream, ta, tb, C, g);
}

int check_gemm(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K) {
    if (M < 0 || N <= 0 || K <= 0) return BIV_ERR_SHAPE;
    if (N % 8 != 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (out_dtype != BIV_BF16 && out_dtype != BIV_F32) return BIV_ERR_VALUE;
    if (M == 0) return BIV_OK;
    if (!A || !B || !C) return BIV_ERR_NULL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return BIV_ERR_ALIGN;
    return BIV_OK;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" int biv_gemm_tile_n(int M, int N, int K) {
    (void)K;
    const long long m_tiles = std::max<long long>(1, ceil_div(M, kBM));
    if (m_tiles == 1) {
        // Weight streaming: one wave of tiles, each as wide as that allows.
        const int bn = static_cast<int>(std::min<long long>(256, std::max<long long>(16, ceil_div(ceil_div(N, kWave), 16) * 16)));
        if (ceil_div(N, bn) <= kWave) return bn;
    }
    // Several waves: the width in [64, 256] that best fills the waves, with a
    // mild preference for wide tiles (less activation traffic per weight byte).
    int best = 256;
    double best_score = -1.0;
    for (int bn = 256; bn >= 64; bn -= 16) {
        const long long tiles = m_tiles * ceil_div(N, bn);
        const long long waves = ceil_div(tiles, kWave);
        const double fill = static_cast<double>(tiles) / static_cast<double>(waves * kWave);
        const double score = fill * bn / (bn + 32.0);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = bn;
        }
    }
    return best;
}

extern "C" int biv_gemm_nosplitk_bn(const void* A, const void* B, void* C, int out_dtype, int M, int N,
                                    int K, int bn, biv_stream_t stream) {
    int st = check_gemm(A, B, C, out_dtype, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    if (bn < 16 || bn > 256 || bn % 16 != 0) return BIV_ERR_VALUE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return out_dtype == BIV_F32 ? launch_gemm<true>(A, B, C, M, N, K, bn, s)
                                : launch_gemm<false>(A, B, C, M, N, K, bn, s);
}

extern "C" int biv_gemm_nosplitk(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K,
                                 biv_stream_t stream) {
    int st = check_gemm(A, B, C, out_dtype, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    return biv_gemm_nosplitk_bn(A, B, C, out_dtype, M, N, K, biv_gemm_tile_n(M, N, K), stream);
}
