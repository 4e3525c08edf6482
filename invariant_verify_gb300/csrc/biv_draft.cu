// Training-free n-gram lookup drafter (NVIDIA inference guide page: among the
// drafting methods it lists, one needs no training and works by finding and
// copying repeated fragments of the earlier text).
//
// For request r with committed history h[0..L): the longest n in
// [n_min, n_max] whose last-n-token suffix also occurs earlier with at least
// one token after it; of those occurrences the most recent (largest start
// p <= L - n - 1).  The drafts copy what followed it, s = p + n:
// d_j = e[s + j], where e is the history with the drafts appended -- a copy
// that runs past the end continues from its own output, as an LZ77 copy
// does, so a periodic text is continued exactly.  No match: all K drafts are
// h[L - 1] (0 for an empty history).  Drafts only steer how many tokens a
// verify step can accept; with coupled Gumbel selection the committed tokens
// do not depend on them.
//
// One CTA per request; for each n from n_max down, the threads test all
// start positions in parallel and the CTA keeps the largest match.
#include <algorithm>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_draft_err)

constexpr int kDraftThreads = 256;
constexpr int kMaxNgram = 64;
constexpr int kMaxDrafts = 1024;

__global__ void __launch_bounds__(kDraftThreads)
ngram_draft_kernel(const int32_t* __restrict__ hist, long long ld, const int32_t* __restrict__ len, int n_max,
                   int n_min, int K, int32_t* __restrict__ drafts, int32_t* __restrict__ draft_src) {
    __shared__ int32_t suffix[kMaxNgram];
    __shared__ int red[kDraftThreads / 32];
    __shared__ int found;
    pdl_wait();
    pdl_trigger();
    const long long r = blockIdx.x;
    const int32_t* h = hist + r * ld;
    int L = len[r];
    if (L < 0 || L > ld) {
        if (threadIdx.x == 0) atomicOr(&g_draft_err, BIV_DEVERR_INDEX);
        L = L < 0 ? 0 : static_cast<int>(ld);
    }
    int src = -1;
    for (int n = n_max; n >= n_min; --n) {
        if (L < n + 1) continue;                       // uniform across the CTA
        __syncthreads();                               // previous n is done with suffix / red
        if (threadIdx.x < n) suffix[threadIdx.x] = h[L - n + threadIdx.x];
        __syncthreads();
        int mine = -1;
        for (int p = threadIdx.x; p <= L - n - 1; p += kDraftThreads) {
            bool match = true;
            for (int i = 0; i < n && match; ++i) match = h[p + i] == suffix[i];
            if (match) mine = p;                       // increasing p: the thread's latest
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine = max(mine, __shfl_xor_sync(0xffffffffu, mine, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mine;
        __syncthreads();
        if (threadIdx.x == 0) {
            int b = -1;
            for (int w = 0; w < kDraftThreads / 32; ++w) b = max(b, red[w]);
            found = b;
        }
        __syncthreads();
        if (found >= 0) {
            src = found + n;
            break;
        }
    }
    if (threadIdx.x == 0) {
        int32_t* d = drafts + r * K;
        for (int j = 0; j < K; ++j) {
            int32_t t;
            if (src < 0) {
                t = L > 0 ? h[L - 1] : 0;
            } else {
                const int i = src + j;
                t = i < L ? h[i] : d[i - L];               // a draft this thread wrote already
            }
            d[j] = t;
        }
        draft_src[r] = src;
    }
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" int biv_ngram_draft(const int32_t* hist, int N, long long ld, const int32_t* len, int n_max, int n_min,
                               int K, int32_t* drafts, int32_t* draft_src, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (N < 0 || ld < 1 || K < 1 || K > kMaxDrafts) return BIV_ERR_SHAPE;
    if (n_min < 1 || n_max < n_min || n_max > kMaxNgram) return BIV_ERR_VALUE;
    if (N == 0) return BIV_OK;
    if (!hist || !len || !drafts || !draft_src) return BIV_ERR_NULL;
    return launch_pdl(ngram_draft_kernel, dim3(static_cast<unsigned>(N)), dim3(kDraftThreads), 0,
                      reinterpret_cast<cudaStream_t>(stream), hist, ld, len, n_max, n_min, K, drafts, draft_src);
}
