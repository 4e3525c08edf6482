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
//   warp 0      TMA producer: per stage one box of A [a_rows x KS*64] and one of
//               B [BN x KS*64] (3-D tensor maps: KS k-blocks of 64 per box; the
//               TMA unit spends a fixed ~275 ns per box whatever its size, so
//               weight-streaming tiles take as many k-blocks per box as two
//               stages allow), 128-byte swizzle, mbarrier transaction counts.  For M <= 128 only the real rows of A are
//               copied (a_rows = M rounded up to 8) and packed back to back;
//               the MMA still reads 128 rows per k-block, and the rows past
//               a_rows hold unrelated data -- harmless, because each row of the
//               product depends only on its own row of A and rows >= M are
//               never stored.
//   warp 1      TMEM allocator + single-thread MMA issuer; commits free smem
//               stages and publish finished accumulators.
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 16 columns, convert, store.
// Two accumulators in TMEM let the epilogue of tile i overlap the MMAs of
// tile i + 1.  Launched with programmatic dependent launch: barrier set-up
// and TMEM allocation overlap the previous kernel.  Every wait is
// bounded (2 s); on time-out the kernel raises BIV_DEVERR_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_gemm_err)

constexpr int kBM = 128;
constexpr int kBK = 64;                       // 64 bf16 = one 128-byte swizzle row
constexpr int kRowBytes = kBK * 2;            // one 64-wide k-block row: 128 B
constexpr int kRingBudget = 208 * 1024;       // bytes of pipeline stages per CTA
constexpr int kTailSlack = kBM * kRowBytes;   // the MMA may read 128 A rows past the last stage
constexpr int kMaxStages = 24;
constexpr int kBarBytes = 512;
constexpr int kWave = 152;                    // CTAs of one wave on a 152-SM part

struct GemmArgs {
    int M, N, K;
    int BN;          // tile width (multiple of 16, 16..256)
    int KS;          // 64-wide k-blocks per stage (one TMA box each for A and B)
    int KB;          // k-blocks in K
    int three_d;     // 3-D tensor maps (K % 64 == 0), else 2-D with KS = 1
    int stages;      // ring depth
    int a_rows;      // rows of A copied per k-block (multiple of 8, <= 128)
    uint32_t idesc;  // tcgen05 instruction descriptor for M=128, N=BN
    uint32_t tmem_cols;
};

inline int stage_bytes(int KS, int a_rows, int BN) { return KS * (a_rows + BN) * kRowBytes; }

// EPI: 0 = bf16 C, 1 = fp32 C, 2 = SwiGLU of gate/up-interleaved B (bf16
// activation [M, N/2]; see biv_gemm_swiglu).
template <int EPI>
__global__ void __launch_bounds__(192, 1)
gemm_nosplitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     void* __restrict__ C, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int A_BYTES = g.KS * g.a_rows * kRowBytes;     // A region of a stage
    const int STAGE = A_BYTES + g.KS * g.BN * kRowBytes;
    const int S = g.stages;
    uint8_t* tiles = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE + (g.a_rows < kBM ? kTailSlack : 0));
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
    const int KB = g.KB;
    const int KS = g.KS;
    const int n_stage_blocks = (KB + KS - 1) / KS;        // stages per tile
    const uint32_t tx_bytes = static_cast<uint32_t>(STAGE);

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
                for (int sb = 0; sb < n_stage_blocks; ++sb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_gemm_err, true)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = tiles + stage * STAGE;
                    mbar_arrive_expect_tx(&full[stage], tx_bytes);
                    if (g.three_d) {
                        tma_load_3d(sa, &tmA, &full[stage], 0, m_blk * kBM, sb * KS, pol_a);
                        tma_load_3d(sa + A_BYTES, &tmB, &full[stage], 0, n_blk * BN, sb * KS, pol_b);
                    } else {
                        tma_load_2d(sa, &tmA, &full[stage], sb * kBK, m_blk * kBM, pol_a);
                        tma_load_2d(sa + A_BYTES, &tmB, &full[stage], sb * kBK, n_blk * BN, pol_b);
                    }
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
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, &g_gemm_err, true)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int sb = 0; sb < n_stage_blocks; ++sb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, &g_gemm_err, true)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + stage * STAGE);
                    const uint32_t b_addr = a_addr + static_cast<uint32_t>(A_BYTES);
                    for (int j = 0; j < KS; ++j) {
                        const int kb = sb * KS + j;
                        if (kb >= KB) break;
                        const uint64_t a_desc = sw128_kmajor_desc(a_addr + static_cast<uint32_t>(j * g.a_rows * kRowBytes));
                        const uint64_t b_desc = sw128_kmajor_desc(b_addr + static_cast<uint32_t>(j * BN * kRowBytes));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // +32 bytes along K inside the swizzle row = +2 in 16-byte units.
                            umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, g.idesc, (kb > 0 || k > 0) ? 1u : 0u);
                        }
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
            if constexpr (EPI == 2) {
                // Columns [32j, 32j + 16) of the tile are gate rows, [32j + 16, 32j + 32)
                // the matching up rows: act = bf16(silu(bf16(g)) * bf16(u)).
                const int F = N / 2;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t gr[16], ur[16];
                    tmem_ld16(taddr + static_cast<uint32_t>(c), gr);
                    tmem_ld16(taddr + static_cast<uint32_t>(c + 16), ur);
                    tmem_ld_wait();
                    const int col = n_blk * BN + c;
                    if (row < M && col < N) {
                        uint32_t o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = swiglu_pack(pack_bf16x2(__uint_as_float(gr[2 * e]), __uint_as_float(gr[2 * e + 1])),
                                               pack_bf16x2(__uint_as_float(ur[2 * e]), __uint_as_float(ur[2 * e + 1])));
                        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(C) +
                                                              static_cast<long long>(row) * F + col / 2);
                        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            } else {
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
                            if constexpr (EPI == 1) {
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

// Row-major bf16 [rows, cols] viewed by TMA with 128-B swizzle.  2-D: boxes of
// [box_rows x 64].  3-D (cols % 64 == 0): the view [cols/64][rows][64] (k-block,
// row, column; strides 128 B and cols*2 B), boxes of [ks][box_rows][64], so
// one box brings ks consecutive k-blocks, each a [box_rows x 64] swizzled tile.
bool encode_kmajor(CUtensorMap* map, const void* base, int cols, int rows, int box_rows, int ks, bool three_d) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    CUresult r;
    if (!three_d) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
        cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
        cuuint32_t estr[2] = {1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, 128};
        cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(ks)};
        cuuint32_t estr[3] = {1, 1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

uint32_t tmem_cols_for(int BN) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(2 * BN)) c <<= 1;
    return c;
}

template <int EPI>
int launch_gemm(const void* A, const void* B, void* C, int M, int N, int K, int BN, cudaStream_t stream) {
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.BN = BN;
    g.a_rows = M >= kBM ? kBM : ((M + 7) / 8) * 8;
    g.KB = (K + kBK - 1) / kBK;
    g.three_d = (K % kBK == 0) ? 1 : 0;
    // The TMA unit spends a fixed ~275 ns per box whatever its size, so a box
    // should be as large as possible.  With one row tile (M <= 128, weight
    // streaming) each stage takes as many k-blocks as let two stages fit the
    // ring; the MMA may then read past the packed A rows of the last stage, so
    // the ring keeps a tail.  Otherwise (full 128-row tiles, compute-bound) one
    // k-block per stage and as many stages as fit.
    int ks = 1;
    const int tail = g.a_rows < kBM ? kTailSlack : 0;
    if (g.three_d && g.a_rows < kBM) {
        const int per_kb = (g.a_rows + BN) * kRowBytes;
        ks = std::max(1, (kRingBudget - tail) / (2 * per_kb));
        ks = std::min(ks, std::min(g.KB, 256));
    }
    g.KS = ks;
    g.stages = std::min(kMaxStages, std::max(1, (kRingBudget - tail) / stage_bytes(ks, g.a_rows, BN)));
    g.idesc = idesc_bf16_f32(kBM, BN);
    g.tmem_cols = tmem_cols_for(BN);
    CUtensorMap ta, tb;
    if (!encode_kmajor(&ta, A, K, M, g.a_rows, ks, g.three_d) || !encode_kmajor(&tb, B, K, N, BN, ks, g.three_d)) {
        set_cuda_error(cudaErrorInvalidValue);
        return BIV_ERR_CUDA;
    }
    const int smem = 1024 + g.stages * stage_bytes(ks, g.a_rows, BN) + tail + kBarBytes;
    auto kern = gemm_nosplitk_kernel<EPI>;
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

// Packed row p: block j = p / 32; rows 32j..32j+15 are gate rows 16j..16j+15,
// rows 32j+16..32j+31 the up rows 16j..16j+15 (source: F gate rows, then F up rows).
__global__ void swiglu_pack_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int F,
                                   int K) {
    pdl_wait();
    pdl_trigger();
    const long long p = blockIdx.x;
    const int j = static_cast<int>(p / 32), r = static_cast<int>(p % 32);
    const long long s = r < 16 ? 16LL * j + r : static_cast<long long>(F) + 16LL * j + (r - 16);
    const uint4* in = reinterpret_cast<const uint4*>(src + s * K);
    uint4* out = reinterpret_cast<uint4*>(dst + p * K);
    for (int c = threadIdx.x; c < K / 8; c += blockDim.x) out[c] = in[c];
}

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
    return out_dtype == BIV_F32 ? launch_gemm<1>(A, B, C, M, N, K, bn, s)
                                : launch_gemm<0>(A, B, C, M, N, K, bn, s);
}

extern "C" int biv_gemm_nosplitk(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K,
                                 biv_stream_t stream) {
    int st = check_gemm(A, B, C, out_dtype, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    return biv_gemm_nosplitk_bn(A, B, C, out_dtype, M, N, K, biv_gemm_tile_n(M, N, K), stream);
}

extern "C" int biv_swiglu_pack_weights(const void* w_gu, void* w_packed, int F, int K, biv_stream_t stream) {
    if (F <= 0 || K <= 0 || F % 16 != 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (!w_gu || !w_packed) return BIV_ERR_NULL;
    if (!aligned16(w_gu) || !aligned16(w_packed)) return BIV_ERR_ALIGN;
    if (w_gu == w_packed) return BIV_ERR_VALUE;
    return launch_pdl(swiglu_pack_kernel, dim3(2 * F), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(w_gu), static_cast<__nv_bfloat16*>(w_packed), F, K);
}

extern "C" int biv_gemm_swiglu(const void* A, const void* B_packed, void* act, int M, int F, int K,
                               biv_stream_t stream) {
    if (F <= 0 || F % 16 != 0) return BIV_ERR_SHAPE;
    const int N = 2 * F;
    int st = check_gemm(A, B_packed, act, BIV_BF16, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    const int bn = static_cast<int>(std::min<long long>(256, ceil_div(biv_gemm_tile_n(M, N, K), 32) * 32));
    return launch_gemm<2>(A, B_packed, act, M, N, K, bn, reinterpret_cast<cudaStream_t>(stream));
}
