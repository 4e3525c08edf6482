// Row-wise kernels: RMSNorm with a fixed reduction shape, and the per-row
// glue of the decoder layer (embedding gather, SwiGLU, residual add).
//
// [DVR] para 1: batch-invariant RMSNorm splits the hidden dimension in a fixed
// way that does not depend on the number of rows or of busy SMs.  Here one
// CTA owns one row; the CTA size is a function of d only; thread t owns the
// 8-element chunks t, t + nthreads, ...; each thread sums its squares in that
// order, the warp combines with a fixed xor butterfly, and warp 0 adds the
// warp partials in increasing warp order.
#include <algorithm>
#include <cmath>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_rowops_err)

constexpr int kMaxChunksPerThread = 2;

int rms_threads(int d) {
    const int chunks = d / 8;
    int t = std::min(chunks, 1024);
    return (t + 31) / 32 * 32;
}

// MODE 0: y = rmsnorm(x).  MODE 1: x_out = bf16(x + r), y = rmsnorm(x_out).
// MODE 2: x_out = table[tokens[row]], y = rmsnorm(x_out).  The norm always
// reads the bf16 row it stores, with the same chunking and reduction tree, so
// the fused modes give the same bits as the separate kernels.
template <int MODE>
__global__ void rmsnorm_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ r,
                               const int32_t* __restrict__ tokens, int vocab, const __nv_bfloat16* __restrict__ w,
                               __nv_bfloat16* __restrict__ x_out, __nv_bfloat16* __restrict__ y, int d, float eps) {
    __shared__ float warp_part[32];
    pdl_wait();
    pdl_trigger();
    const long long row = blockIdx.x;
    const int chunks = d / 8;
    const uint4* xr;
    if constexpr (MODE == 2) {
        int tok = tokens[row];
        if (tok < 0 || tok >= vocab) {
            if (threadIdx.x == 0) atomicOr(&g_rowops_err, BIV_DEVERR_INDEX);
            tok = -1;
        }
        xr = reinterpret_cast<const uint4*>(x + static_cast<long long>(tok < 0 ? 0 : tok) * d);
        if (tok < 0) xr = nullptr;
    } else {
        xr = reinterpret_cast<const uint4*>(x + row * d);
    }
    uint4 v[kMaxChunksPerThread];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kMaxChunksPerThread; ++k) {
        const int c = threadIdx.x + k * blockDim.x;
        v[k] = make_uint4(0, 0, 0, 0);
        if (c < chunks) {
            if constexpr (MODE == 1) {
                const uint4 a = xr[c];
                const uint4 b = reinterpret_cast<const uint4*>(r + row * d)[c];
                const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[e] = pack_bf16x2(__fadd_rn(bf16lo(aa[e]), bf16lo(bb[e])), __fadd_rn(bf16hi(aa[e]), bf16hi(bb[e])));
                v[k] = make_uint4(o[0], o[1], o[2], o[3]);
            } else if constexpr (MODE == 2) {
                if (xr) v[k] = xr[c];
            } else {
                v[k] = xr[c];
            }
            const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float a = bf16lo(u[e]), b = bf16hi(u[e]);
                ss = __fmaf_rn(a, a, ss);
                ss = __fmaf_rn(b, b, ss);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) warp_part[warp] = ss;
    __syncthreads();
    if (warp == 0) {
        float t = 0.0f;
        const int nw = blockDim.x >> 5;
        if (lane == 0) {
            for (int i = 0; i < nw; ++i) t += warp_part[i];
            warp_part[0] = t;
        }
    }
    __syncthreads();
    const float inv = rsqrtf(__fadd_rn(__fdiv_rn(warp_part[0], static_cast<float>(d)), eps));
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    uint4* yr = reinterpret_cast<uint4*>(y + row * d);
#pragma unroll
    for (int k = 0; k < kMaxChunksPerThread; ++k) {
        const int c = threadIdx.x + k * blockDim.x;
        if (c < chunks) {
            if constexpr (MODE != 0) reinterpret_cast<uint4*>(x_out + row * d)[c] = v[k];
            const uint4 g = wr[c];
            const uint32_t u[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = pack_bf16x2(__fmul_rn(__fmul_rn(bf16lo(u[e]), inv), bf16lo(gw[e])),
                                   __fmul_rn(__fmul_rn(bf16hi(u[e]), inv), bf16hi(gw[e])));
            yr[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

__global__ void embed_kernel(const __nv_bfloat16* __restrict__ table, const int32_t* __restrict__ tokens,
                             __nv_bfloat16* __restrict__ out, int d, int vocab) {
    pdl_wait();
    pdl_trigger();
    const long long w = blockIdx.x;
    const int tok = tokens[w];
    uint4* dst = reinterpret_cast<uint4*>(out + w * d);
    const bool ok = tok >= 0 && tok < vocab;
    if (!ok && threadIdx.x == 0) atomicOr(&g_rowops_err, BIV_DEVERR_INDEX);
    const uint4* src = reinterpret_cast<const uint4*>(table + static_cast<long long>(ok ? tok : 0) * d);
    for (int c = threadIdx.x; c < d / 8; c += blockDim.x) dst[c] = ok ? src[c] : make_uint4(0, 0, 0, 0);
}

__global__ void silu_mul_kernel(const __nv_bfloat16* __restrict__ gu, __nv_bfloat16* __restrict__ out, int rows,
                                int F) {
    pdl_wait();
    pdl_trigger();
    const long long per_row = F / 8;
    const long long total = static_cast<long long>(rows) * per_row;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = i / per_row, c = i - r * per_row;
        const uint4 g = reinterpret_cast<const uint4*>(gu + r * 2 * F)[c];
        const uint4 u = reinterpret_cast<const uint4*>(gu + r * 2 * F + F)[c];
        const uint32_t gg[4] = {g.x, g.y, g.z, g.w}, uu[4] = {u.x, u.y, u.z, u.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[e] = swiglu_pack(gg[e], uu[e]);
        reinterpret_cast<uint4*>(out + r * F)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void residual_add_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ y,
                                    __nv_bfloat16* __restrict__ out, long long n8) {
    pdl_wait();
    pdl_trigger();
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const uint4 a = reinterpret_cast<const uint4*>(x)[i];
        const uint4 b = reinterpret_cast<const uint4*>(y)[i];
        const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            o[e] = pack_bf16x2(__fadd_rn(bf16lo(aa[e]), bf16lo(bb[e])), __fadd_rn(bf16hi(aa[e]), bf16hi(bb[e])));
        reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// One thread waits on a barrier that nothing completes: the library's bounded
// wait gives up after its time limit, raises BIV_DEVERR_TIMEOUT in this
// module's error word and the kernel returns with the context intact.
__global__ void wait_timeout_kernel() {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
        mbar_wait(&bar, 0u, &abort_flag, &g_rowops_err);
    }
}

int grid_for(long long work, int threads) {
    return static_cast<int>(std::max<long long>(1, std::min<long long>((work + threads - 1) / threads,
                                                                       static_cast<long long>(num_sms()) * 16)));
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" int biv_rmsnorm(const void* x, const void* w, void* y, int rows, int d, float eps,
                           biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (rows < 0 || d < 8 || d % 8 != 0 || d > 8 * 1024 * kMaxChunksPerThread) return BIV_ERR_SHAPE;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return BIV_ERR_VALUE;
    if (rows == 0) return BIV_OK;
    if (!x || !w || !y) return BIV_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return BIV_ERR_ALIGN;
    return launch_pdl(rmsnorm_kernel<0>, dim3(rows), dim3(rms_threads(d)), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(nullptr),
                      static_cast<const int32_t*>(nullptr), 0, static_cast<const __nv_bfloat16*>(w),
                      static_cast<__nv_bfloat16*>(nullptr), static_cast<__nv_bfloat16*>(y), d, eps);
}

extern "C" int biv_add_rmsnorm(const void* x, const void* r, const void* w, void* x_out, void* y, int rows, int d,
                               float eps, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (rows < 0 || d < 8 || d % 8 != 0 || d > 8 * 1024 * kMaxChunksPerThread) return BIV_ERR_SHAPE;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return BIV_ERR_VALUE;
    if (rows == 0) return BIV_OK;
    if (!x || !r || !w || !x_out || !y) return BIV_ERR_NULL;
    if (!aligned16(x) || !aligned16(r) || !aligned16(w) || !aligned16(x_out) || !aligned16(y)) return BIV_ERR_ALIGN;
    return launch_pdl(rmsnorm_kernel<1>, dim3(rows), dim3(rms_threads(d)), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(r),
                      static_cast<const int32_t*>(nullptr), 0, static_cast<const __nv_bfloat16*>(w),
                      static_cast<__nv_bfloat16*>(x_out), static_cast<__nv_bfloat16*>(y), d, eps);
}

extern "C" int biv_embed_rmsnorm(const void* table, const int32_t* tokens, const void* w, void* x_out, void* y,
                                 int W, int d, int vocab, float eps, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || d < 8 || d % 8 != 0 || d > 8 * 1024 * kMaxChunksPerThread || vocab <= 0) return BIV_ERR_SHAPE;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return BIV_ERR_VALUE;
    if (W == 0) return BIV_OK;
    if (!table || !tokens || !w || !x_out || !y) return BIV_ERR_NULL;
    if (!aligned16(table) || !aligned16(w) || !aligned16(x_out) || !aligned16(y)) return BIV_ERR_ALIGN;
    return launch_pdl(rmsnorm_kernel<2>, dim3(W), dim3(rms_threads(d)), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(table), static_cast<const __nv_bfloat16*>(nullptr), tokens,
                      vocab, static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(x_out),
                      static_cast<__nv_bfloat16*>(y), d, eps);
}

extern "C" int biv_embed(const void* table, const int32_t* tokens, void* out, int W, int d, int vocab,
                         biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || d <= 0 || d % 8 != 0 || vocab <= 0) return BIV_ERR_SHAPE;
    if (W == 0) return BIV_OK;
    if (!table || !tokens || !out) return BIV_ERR_NULL;
    if (!aligned16(table) || !aligned16(out)) return BIV_ERR_ALIGN;
    return launch_pdl(embed_kernel, dim3(W), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(table), tokens, static_cast<__nv_bfloat16*>(out), d, vocab);
}

extern "C" int biv_silu_mul(const void* gu, void* out, int rows, int F, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (rows < 0 || F <= 0 || F % 8 != 0) return BIV_ERR_SHAPE;
    if (rows == 0) return BIV_OK;
    if (!gu || !out) return BIV_ERR_NULL;
    if (!aligned16(gu) || !aligned16(out)) return BIV_ERR_ALIGN;
    const long long work = static_cast<long long>(rows) * (F / 8);
    return launch_pdl(silu_mul_kernel, dim3(grid_for(work, 256)), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(gu), static_cast<__nv_bfloat16*>(out), rows, F);
}

extern "C" int biv_residual_add(const void* x, const void* y, void* out, long long n, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (n < 0 || n % 8 != 0) return BIV_ERR_SHAPE;
    if (n == 0) return BIV_OK;
    if (!x || !y || !out) return BIV_ERR_NULL;
    if (!aligned16(x) || !aligned16(y) || !aligned16(out)) return BIV_ERR_ALIGN;
    return launch_pdl(residual_add_kernel, dim3(grid_for(n / 8, 256)), dim3(256), 0,
                      reinterpret_cast<cudaStream_t>(stream), static_cast<const __nv_bfloat16*>(x),
                      static_cast<const __nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(out), n / 8);
}

extern "C" int biv_selftest_wait_timeout(biv_stream_t stream) {
    BIV_TRACE_CALL();
    biv::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        biv::set_cuda_error(e);
        return BIV_ERR_CUDA;
    }
    return BIV_OK;
}
