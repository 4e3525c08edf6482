// Seeded Gumbel-max token selection and the coupled accept / rollback check.
//
// [COUPLING] (AIexTime post 185): adding Gumbel(0,1) noise to the logits and
// taking the argmax samples from the softmax without computing one; the
// noise is independent of the logits, and when drafter and target share it
// the verifier only compares two tokens.  Here the noise of vocabulary entry
// v at position p of request r is a pure function of (seed, r, p, v) built
// from Philox4x32-10 (Salmon et al., SC'11), a fixed uniform map and an fp32
// log made only of IEEE +, -, *, /, fma -- so a row gets the same token at
// any batch size, on any machine that follows the same operation sequence.
//
// Selection kernel: one thread-block cluster of 8 CTAs per row.  Each CTA
// stages a contiguous slice of the row in shared memory with bulk async
// copies (one pass over HBM) and finds the winner of its slice; rank 0 takes
// the largest of the 8 slice winners.  Within a slice, candidates are pruned
// exactly in two levels, each against a key that some entry of the slice
// really has (so the slice winner's key is >= the bound):
//   0. LB = the exact key of the slice's largest logit;
//   1. a group of 4 logits (one Philox call) is dropped when even the largest
//      noise cannot lift it to LB: fl(fl(max4 * invT) + 17) < LB -- every
//      noise value is < 17 (the noise lies in [-2.82, 16.64]);
//   2. for the rest, the Philox words are drawn and each entry gets the bound
//      fl(fl(x * invT) + T[w >> 24]), where T[b] bounds the noise of uniform
//      bucket b from above (the noise is a non-decreasing function of the
//      23-bit uniform index, checked over all 2^23 values, so the noise at the
//      bucket's top plus a margin far above the log's error bounds the whole
//      bucket; a GPU test checks every one of the 2^23 noise values against
//      it); the best-bounded entry is evaluated exactly and the larger of its
//      key and LB becomes LB2; only entries whose bound reaches LB2 get their
//      two logs.
// Each CTA also raises its peers' copies of a shared bound (a remote atomic
// max in DSMEM) to every real key it evaluates for LB and LB2, and prunes
// against the larger of its own and the shared one -- on a peaked row the
// slice holding the peak prunes every other slice.  The cluster meets at
// start-up (every CTA's barriers exist before any remote operation), and every
// CTA arrives on a cluster barrier after its last remote bound and waits on
// it before leaving, so no CTA exits while a peer may still write to it.  At
// the end each CTA stores its winner into rank 0's shared memory and arrives
// on rank 0's barrier.
// Rounding is monotone, so no dropped entry can reach the bound.  The winner
// is the maximum of a 64-bit packed value (order(key) << 32 | ~v), which puts
// larger keys first and lower indices first among equal keys, so any
// reduction order gives the same token.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "biv_common.cuh"
#include "biv_gumbel.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_select_err)

constexpr int kClusterSize = 8;
constexpr int kSelThreads = 256;
constexpr int kPieces = 4;
constexpr int kMaxSliceFloats = 45872;          // 5 bytes per logit (value + group bound) <= 224 KiB
constexpr float kNoiseBound = 17.0f;

// Upper bounds of the noise per uniform bucket (top 8 bits of the 23-bit
// uniform index), passed to the kernel by value.
struct NoiseBounds {
    float v[256];
};

// Bucket b holds indices k in [b * 2^15, (b + 1) * 2^15); its largest uniform
// is u = (2 k_max + 1) 2^-24.  Bound = -ln(-ln u) in double + 1e-3, rounded up
// to float: the fp32 noise routine is within a few ulp of the exact value.
const NoiseBounds& noise_bounds() {
    static NoiseBounds nb = [] {
        NoiseBounds t;
        for (int b = 0; b < 256; ++b) {
            const double k = static_cast<double>((b << 15) | 0x7fff);
            const double u = (2.0 * k + 1.0) * 5.9604644775390625e-8;
            const double g = -std::log(-std::log(u)) + 1e-3;
            float f = static_cast<float>(g);
            if (static_cast<double>(f) < g) f = std::nextafter(f, INFINITY);
            t.v[b] = f;
        }
        return t;
    }();
    return nb;
}

// Inverse of key_order for orders of numbers (order 0, NaN, maps to NaN).
BIV_DEV float order_to_float(uint32_t o) {
    return o == 0u ? __int_as_float(0x7fc00000) : __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// ------------------------------------------------------------- cluster PTX
BIV_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

BIV_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
BIV_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

BIV_DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

BIV_DEV void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Block-wide max of a packed value; every thread gets the result.
BIV_DEV unsigned long long block_max64(unsigned long long v, unsigned long long* scratch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_max64(v);
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    unsigned long long r = 0;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; ++w) r = umax64(r, scratch[w]);
    __syncthreads();
    return r;
}

// Remote (cluster) store of a 64-bit value and a release-arrive on a remote
// mbarrier: CTA `rank`'s copy of the shared variable at `local_addr`.
BIV_DEV uint32_t dsmem_addr(const void* local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_addr)), "r"(rank));
    return remote;
}

BIV_DEV void push_to_rank(unsigned long long* slot, uint64_t* bar, uint32_t rank, unsigned long long v) {
    const uint32_t rs = dsmem_addr(slot, rank), rb = dsmem_addr(bar, rank);
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(rs), "l"(v) : "memory");
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rb) : "memory");
}

// Raise every cluster CTA's copy of `slot` to at least v (relaxed remote max).
BIV_DEV void share_bound(unsigned long long* slot, unsigned long long v) {
#pragma unroll 1
    for (uint32_t r = 0; r < kClusterSize; ++r)
        asm volatile("red.shared::cluster.max.u64 [%0], %1;" ::"r"(dsmem_addr(slot, r)), "l"(v) : "memory");
}

BIV_DEV bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------ the kernel
// grid.x = kClusterSize * R, cluster (kClusterSize, 1, 1).  CTA `rank` of the
// cluster owns logits [rank * slice, min((rank + 1) * slice, V)) of row
// blockIdx.x / kClusterSize; slice is a multiple of 4.  Each CTA prunes
// against lower bounds of its own slice (any real key is a valid bound for
// the whole row) and pushes its slice winner into rank 0, which reduces.
__global__ void __launch_bounds__(kSelThreads)
gumbel_argmax_kernel(const float* __restrict__ logits, int V, long long ld, int slice,
                     const uint32_t* __restrict__ row_req, const int32_t* __restrict__ row_pos,
                     uint32_t seed_lo, uint32_t seed_hi, float invT, int greedy,
                     int32_t* __restrict__ tokens, const __grid_constant__ NoiseBounds nb) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float* xs = reinterpret_cast<float*>(smem_raw);
    uint32_t* gub = reinterpret_cast<uint32_t*>(smem_raw + static_cast<size_t>(slice) * 4);  // per group
    __shared__ uint64_t bars[kPieces];
    __shared__ uint64_t inbox_bar;                             // rank 0: one arrival per CTA
    __shared__ unsigned long long inbox[kClusterSize];         // rank 0: slice winners
    __shared__ unsigned long long red[kSelThreads / 32];
    __shared__ unsigned long long bcast;
    __shared__ unsigned long long lb_all;                      // largest real key any CTA of the row has found
    __shared__ float gtab[256];                                // noise bound of each uniform bucket
    __shared__ int abort_flag;

    static_assert(kSelThreads == 256, "one bucket per thread");
    const uint32_t rank = cluster_rank();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        lb_all = 0;
        for (int p = 0; p < kPieces; ++p) mbar_init(&bars[p], 1);
        mbar_init(&inbox_bar, kClusterSize);
        fence_mbar_init();
    }
    gtab[threadIdx.x] = nb.v[threadIdx.x];
    cluster_sync();           // every CTA's barriers exist before any remote arrive
    pdl_wait();
    pdl_trigger();

    const long long row = blockIdx.x / kClusterSize;
    const int begin = static_cast<int>(rank) * slice;
    const int count = max(0, min(slice, V - begin));          // multiple of 4
    const float* src = logits + row * ld + begin;
    const int piece = ((count / 4 + kPieces - 1) / kPieces) * 4;
    if (threadIdx.x == 0) {
        for (int p = 0; p < kPieces; ++p) {
            const int off = p * piece;
            const int n = max(0, min(piece, count - off));
            mbar_arrive_expect_tx(&bars[p], static_cast<uint32_t>(n) * 4u);
            if (n > 0) bulk_g2s(xs + off, src + off, static_cast<uint32_t>(n) * 4u, &bars[p]);
        }
    }
    const uint32_t req = row_req[row];
    const uint32_t pos = static_cast<uint32_t>(row_pos[row]) + 1u;   // position being selected

    // Pass 1: slice maximum (value, lowest index), piece by piece as it lands.
    float best_x = 0.0f;
    int best_i = -1;
    bool ok = true;
    for (int p = 0; p < kPieces; ++p) {
        if (!mbar_wait(&bars[p], 0, &abort_flag, &g_select_err)) {
            ok = false;
            break;
        }
        const int off = p * piece;
        const int n = max(0, min(piece, count - off));
        for (int i = threadIdx.x * 4; i < n; i += kSelThreads * 4) {
            const float4 v = *reinterpret_cast<const float4*>(xs + off + i);
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x = e[j];
                if (x == x && (best_i < 0 || x > best_x)) {   // NaN never becomes the max
                    best_x = x;
                    best_i = begin + off + i + j;
                }
            }
        }
    }
    unsigned long long mx = best_i >= 0 ? pack_key(best_x, static_cast<uint32_t>(best_i)) : 0ull;
    mx = block_max64(mx, red);
    if (!ok && threadIdx.x == 0)
        for (int p = 0; p < kPieces; ++p) mbar_wait_drain(&bars[p], 0);   // copies in flight land first

    unsigned long long best = mx;
    if (!greedy && ok) {
        // LB: the exact key of this slice's largest logit.
        if (threadIdx.x == 0) {
            unsigned long long lb = 0;
            if (mx) {
                const uint32_t v = ~static_cast<uint32_t>(mx & 0xffffffffull);
                const U4 w = philox4x32_10(v >> 2, pos, req, 0u, seed_lo, seed_hi);
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                lb = pack_key(__fadd_rn(__fmul_rn(xs[v - begin], invT), gumbel_from_word(words[v & 3u])), v);
            }
            bcast = lb;
            share_bound(&lb_all, lb);
        }
        __syncthreads();
        const unsigned long long lb = bcast;
        const uint32_t lb_order = static_cast<uint32_t>(lb >> 32);
        // Any real key of the row bounds its winner, so the bound used below is
        // the larger of this slice's and whatever the other slices have sent.
        const volatile unsigned long long* lbv = &lb_all;

        // Pass A: level-1 pruning, then Philox words and level-2 bounds.
        const int n_groups = count / 4;
        unsigned long long cb = 0;          // best level-2 bound of this thread (order, ~index)
        for (int gi = threadIdx.x; gi < n_groups; gi += kSelThreads) {
            const float4 v4 = *reinterpret_cast<const float4*>(xs + 4 * gi);
            const float m4 = fmaxf(fmaxf(v4.x, v4.y), fmaxf(v4.z, v4.w));
            uint32_t g_ord = 0;
            const uint32_t lbo = max(lb_order, static_cast<uint32_t>(*lbv >> 32));
            if (key_order(__fadd_rn(__fmul_rn(m4, invT), kNoiseBound)) >= lbo) {
                const uint32_t v0 = static_cast<uint32_t>(begin + 4 * gi);
                const U4 w = philox4x32_10(v0 >> 2, pos, req, 0u, seed_lo, seed_hi);
                const float e[4] = {v4.x, v4.y, v4.z, v4.w};
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t o = key_order(__fadd_rn(__fmul_rn(e[j], invT), gtab[words[j] >> 24]));
                    g_ord = max(g_ord, o);
                    cb = umax64(cb, (static_cast<unsigned long long>(o) << 32) |
                                        static_cast<unsigned long long>(~(v0 + j)));
                }
            }
            gub[gi] = g_ord;
        }
        cb = block_max64(cb, red);
        // LB2: the exact key of the best-bounded entry (a real key), or LB.
        if (threadIdx.x == 0) {
            unsigned long long cand = lb;
            if (cb) {
                const uint32_t v = ~static_cast<uint32_t>(cb & 0xffffffffull);
                const U4 w = philox4x32_10(v >> 2, pos, req, 0u, seed_lo, seed_hi);
                const uint32_t words[4] = {w.x, w.y, w.z, w.w};
                cand = umax64(cand, pack_key(__fadd_rn(__fmul_rn(xs[v - begin], invT),
                                                       gumbel_from_word(words[v & 3u])), v));
            }
            bcast = cand;
            share_bound(&lb_all, cand);
        }
        __syncthreads();
        cluster_arrive();         // this CTA sends no more bounds
        const unsigned long long lb2 = bcast;
        const uint32_t lb2_order = static_cast<uint32_t>(lb2 >> 32);

        // Pass B: exact keys only where the level-2 bound reaches LB2.
        best = lb2;
        for (int gi = threadIdx.x; gi < n_groups; gi += kSelThreads) {
            const uint32_t lbo = max(lb2_order, static_cast<uint32_t>(*lbv >> 32));
            if (gub[gi] < lbo) continue;
            const float4 v4 = *reinterpret_cast<const float4*>(xs + 4 * gi);
            const uint32_t v0 = static_cast<uint32_t>(begin + 4 * gi);
            const U4 w = philox4x32_10(v0 >> 2, pos, req, 0u, seed_lo, seed_hi);
            const float e[4] = {v4.x, v4.y, v4.z, v4.w};
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float a = __fmul_rn(e[j], invT);
                if (key_order(__fadd_rn(a, gtab[words[j] >> 24])) < lbo) continue;
                best = umax64(best, pack_key(__fadd_rn(a, gumbel_from_word(words[j])), v0 + j));
            }
        }
        best = block_max64(best, red);
    } else {
        cluster_arrive();
    }

    // The slice winner goes to rank 0; rank 0 waits for all, reduces and stores.
    if (threadIdx.x == 0) push_to_rank(&inbox[rank], &inbox_bar, 0, best);
    if (rank == 0 && threadIdx.x == 0) {
        const uint64_t t0 = globaltimer();
        bool got = true;
        while (!mbar_try_wait_cluster(&inbox_bar, 0)) {
            if (globaltimer() - t0 > kWaitLimitNs) {
                atomicOr(&g_select_err, BIV_DEVERR_TIMEOUT);
                got = false;
                break;
            }
        }
        unsigned long long w = 0;
        if (got)
            for (int c = 0; c < kClusterSize; ++c) w = umax64(w, inbox[c]);
        tokens[row] = w ? static_cast<int32_t>(~static_cast<uint32_t>(w & 0xffffffffull)) : 0;
    }
    cluster_wait();               // no CTA leaves while a peer may still send it a bound
}


// ------------------------------------------------ streaming row kernel
// One CTA per row (persistent over rows), no cross-CTA traffic.  Pass 1
// streams the row from HBM through a ring of kStreamStages bulk copies and
// keeps the maximum of every 256-logit block in shared memory, and the row's
// largest logit.  The exact key of that logit is the lower bound LB.  Pass 2
// lists the blocks whose maximum can still reach LB with the largest noise of
// all, then re-reads (mostly from L2) only their logits, every thread with
// kUnroll loads in flight; per 4-group it draws the Philox words, bounds each
// entry by fl(fl(x * invT) + T[w >> 24]) and takes the two logs only where
// that bound passes the best key found so far.  Entries are skipped only on
// a bound at or below a real key of the row, so the result is exact.  On a
// peaked row pass 2 touches a block or two.  A flat row (most blocks live)
// is bound by the Philox arithmetic, several times a row's streaming time on
// one CTA while the others stream; it is handed off instead, in per-chunk
// units, to a second kernel that runs over all SMs after this one
// (gumbel_units_kernel).  The ring runs ahead across rows: the next row's
// first chunks land during pass 2.
constexpr int kStreamChunk = 8192;               // floats per ring slot (32 KiB)
constexpr int kStreamStages = 2;
constexpr int kBlock = 256;                      // logits per block maximum
constexpr int kMaxStreamV = 1 << 22;             // block maxima kept in shared memory (64 KiB)
constexpr int kUnroll = 4;                       // pass 2: loads in flight per thread
constexpr int kCtrSlots = 64;                    // row-ticket counter pairs, one per launch in flight

// {next row ticket, CTAs finished} per slot; zero at load, and the last CTA of
// every launch puts its pair back to zero.
__device__ unsigned int g_stream_ctr[2 * kCtrSlots];

// Rows whose live blocks are many (flat rows: the noise, not one large logit,
// decides them) are handed from the streaming kernel to the unit kernel,
// which spreads their work over every SM in 32 KiB units (one chunk of the
// row and its live blocks).  Stream-ordered scratch of one call:
struct HeavyRows {
    unsigned int* ctr;         // {heavy slots taken, units registered, unit ticket} (zero at entry)
    unsigned long long* best;  // [cap] the row's best packed key so far (LB at hand-off)
    int* row_of;               // [cap] heavy slot -> row
    int* remaining;            // [cap] units of the row not yet done
    int4* units;               // [cap * n_chunks] (slot, chunk, first, end) into the live list
    uint16_t* live;            // [cap][n_blocks] the row's live blocks, ascending
    int cap;                   // heavy slots; 0 = no hand-off (every row done in place)
    int min_live;              // a row with more live blocks than this is handed off
};

// Pass 2b over n_items 4-groups: item it is group it % 64 of block
// blk_of(it >> 6); entry v is read at src + v - off.  Every thread runs the
// same number of iterations (a CTA-wide running best is shared through
// s_best).  Returns the thread's best packed key.
template <int UNROLL, typename BlkOf>
BIV_DEV unsigned long long groups_pass(const float* src, long long off, int n_items, BlkOf blk_of, int V, uint32_t pos,
                                       uint32_t req, uint32_t seed_lo, uint32_t seed_hi, float invT, const float* gtab,
                                       float g254, unsigned long long best, unsigned long long* s_best) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int base = 0; base < n_items; base += kSelThreads * UNROLL) {
        float4 v4[UNROLL];
        int v0[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int it = base + u * kSelThreads + static_cast<int>(threadIdx.x);
            v0[u] = -1;
            if (it < n_items) {
                const int v = blk_of(it >> 6) * kBlock + 4 * (it & 63);
                if (v < V) {                          // the last block may be partial
                    v0[u] = v;
                    v4[u] = *reinterpret_cast<const float4*>(src + (v - off));
                }
            }
        }
        // Straight-line over the UNROLL groups so their Philox chains
        // interleave.  A bound strictly below best_f (the value of the
        // best key) cannot win; equal or NaN-free ties go to the exact
        // packed comparison.  While best is a NaN key (order 0: a row
        // with no number so far) nothing is pruned.
        const bool no_prune = (best >> 32) == 0;
        const float best_f = order_to_float(static_cast<uint32_t>(best >> 32));
        U4 w[UNROLL];
        bool glive[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const float m4 = fmaxf(fmaxf(v4[u].x, v4[u].y), fmaxf(v4[u].z, v4[u].w));
            glive[u] = v0[u] >= 0 && (no_prune || __fadd_rn(__fmul_rn(m4, invT), kNoiseBound) >= best_f);
            w[u] = philox4x32_10(static_cast<uint32_t>(max(v0[u], 0)) >> 2, pos, req, 0u, seed_lo, seed_hi);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            if (!glive[u]) continue;
            const float e[4] = {v4[u].x, v4[u].y, v4[u].z, v4[u].w};
            const uint32_t words[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            // Below the top byte 255 no noise exceeds g254: if even the
            // group's largest logit cannot pass with it, only entries
            // whose word has top byte 255 need their own bound.
            const float m4 = fmaxf(fmaxf(v4[u].x, v4[u].y), fmaxf(v4[u].z, v4[u].w));
            const bool top_only = !no_prune && __fadd_rn(__fmul_rn(m4, invT), g254) < best_f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (top_only && words[j] < 0xFF000000u) continue;
                const float a = __fmul_rn(e[j], invT);
                if (!no_prune && !(__fadd_rn(a, gtab[words[j] >> 24]) >= best_f)) continue;
                const uint32_t vv = static_cast<uint32_t>(v0[u] + j);
                best = umax64(best, pack_key(__fadd_rn(a, gumbel_from_word(words[j])), vv));
            }
        }
        // share the bound: warp maximum, then the CTA's running maximum
        best = warp_max64(best);
        if (lane == 0) atomicMax(s_best, best);
        best = umax64(best, *reinterpret_cast<volatile unsigned long long*>(s_best));
    }
    return best;
}

// First index i in the ascending list[0 .. n) with list[i] >= key.
BIV_DEV int lower_bound_int(const int* list, int n, int key) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (list[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}


size_t stream_smem_bytes(int V) {
    return static_cast<size_t>(kStreamStages) * kStreamChunk * 4 + static_cast<size_t>((V + kBlock - 1) / kBlock) * 4;
}

__global__ void __launch_bounds__(kSelThreads, 3)
gumbel_stream_kernel(const float* __restrict__ logits, int R, int V, long long ld,
                     const uint32_t* __restrict__ row_req, const int32_t* __restrict__ row_pos, uint32_t seed_lo,
                     uint32_t seed_hi, float invT, int greedy, int32_t* __restrict__ tokens,
                     unsigned int* __restrict__ ctr, const __grid_constant__ NoiseBounds nb, const HeavyRows hv) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float* ring = reinterpret_cast<float*>(smem_raw);                                     // [stages][chunk]
    float* bmax = reinterpret_cast<float*>(smem_raw + kStreamStages * kStreamChunk * 4);  // [ceil(V / 256)]
    __shared__ uint64_t fbar[kStreamStages];
    __shared__ unsigned long long red[kSelThreads / 32];
    __shared__ unsigned long long bcast;
    __shared__ unsigned long long s_best;                    // pass 2: best key any warp has found
    __shared__ int wcount[kSelThreads / 32];
    __shared__ int s_rows[8];                                // row of stream ordinal i at [i % 8]
    __shared__ int s_heavy, s_unit0;                         // hand-off: heavy slot, first unit
    int* live_list = reinterpret_cast<int*>(bmax);           // pass 2: live blocks, written over bmax
    __shared__ float gtab[256];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStreamStages; ++i) mbar_init(&fbar[i], 1);
        fence_mbar_init();
    }
    gtab[threadIdx.x] = nb.v[threadIdx.x];
    const float g254 = nb.v[254];                  // largest noise bound below the top byte 255
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    const int n_chunks = (V + kStreamChunk - 1) / kStreamChunk;
    const int n_blocks = (V + kBlock - 1) / kBlock;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    static_assert(kStreamChunk % kBlock == 0, "blocks never straddle chunks");
    static_assert(kBlock == 256, "pass 2 indexes 64 groups per block");
    // Rows are dealt out by a ticket counter, so a CTA that meets an expensive
    // (flat) row takes fewer rows.  Thread 0 fetches the ticket of a row when
    // it issues the row's first chunk, up to kStreamStages chunks ahead of the
    // consumers, and posts it in s_rows (-1: no rows left); every thread reads
    // it after at least one barrier that follows the post.
    long long k_issued = 0;                          // thread 0: chunks issued
    bool stream_end = false;                         // thread 0: a ticket past the last row came back
    auto issue_next = [&]() {
        if (stream_end) return;
        const long long ord = k_issued / n_chunks;
        const int c = static_cast<int>(k_issued % n_chunks);
        if (c == 0) {
            const unsigned t = atomicAdd(&ctr[0], 1u);
            s_rows[ord & 7] = t < static_cast<unsigned>(R) ? static_cast<int>(t) : -1;
            if (t >= static_cast<unsigned>(R)) {
                stream_end = true;
                return;
            }
        }
        const long long rr = s_rows[ord & 7];
        const int n = min(kStreamChunk, V - c * kStreamChunk);
        const int slot = static_cast<int>(k_issued % kStreamStages);
        mbar_arrive_expect_tx(&fbar[slot], static_cast<uint32_t>(n) * 4u);
        bulk_g2s(ring + slot * kStreamChunk, logits + rr * ld + static_cast<long long>(c) * kStreamChunk,
                 static_cast<uint32_t>(n) * 4u, &fbar[slot]);
        ++k_issued;
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < kStreamStages; ++i) issue_next();
    __syncthreads();

    long long k = 0;                                 // next chunk to consume
    bool ok = true;
#pragma unroll 1
    for (long long ord = 0;; ++ord) {
        const int row = s_rows[ord & 7];
        if (row < 0) break;
        const float* x = logits + static_cast<long long>(row) * ld;
        const uint32_t req = row_req[row];                                 // used after pass 1
        const uint32_t pos = static_cast<uint32_t>(row_pos[row]) + 1u;   // position being selected
        // ---- pass 1: block maxima and the row maximum (lowest index among equals)
        float best_x = 0.0f;
        int best_i = -1;
#pragma unroll 1
        for (int c = 0; c < n_chunks; ++c) {
            const int slot = static_cast<int>(k % kStreamStages);
            mbar_wait(&fbar[slot], static_cast<uint32_t>((k / kStreamStages) & 1), &abort_flag, &g_select_err);
            __syncthreads();                          // a timed-out wait is seen by every thread
            if (abort_flag) {
                ok = false;
                break;
            }
            const int n = min(kStreamChunk, V - c * kStreamChunk);   // a multiple of 4
            const float* buf = ring + slot * kStreamChunk;
            // warp per 256-logit block; lane l reads logits [4l, 4l+4) and [128+4l, 128+4l+4)
#pragma unroll 1
            for (int blk = warp; blk * kBlock < n; blk += kSelThreads / 32) {
                float m = __int_as_float(0x7fc00000);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int e0 = blk * kBlock + h * 128 + 4 * lane;
                    if (e0 >= n) break;
                    const float4 v = *reinterpret_cast<const float4*>(buf + e0);
                    const float m4 = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                    m = fmaxf(m, m4);
                    if (m4 == m4 && (best_i < 0 || m4 > best_x)) {      // lanes see their logits in index order
                        best_x = m4;
                        best_i = c * kStreamChunk + e0 + (v.x == m4 ? 0 : v.y == m4 ? 1 : v.z == m4 ? 2 : 3);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                if (lane == 0) bmax[c * (kStreamChunk / kBlock) + blk] = m;
            }
            __syncthreads();                          // the slot is read; refill it
            if (threadIdx.x == 0) issue_next();
            ++k;
        }
        if (!ok) break;
        unsigned long long mx = best_i >= 0 ? pack_key(best_x, static_cast<uint32_t>(best_i)) : 0ull;
        mx = block_max64(mx, red);
        unsigned long long best = mx;
        if (!greedy) {
            // LB: the exact key of the row's largest logit.
            if (threadIdx.x == 0) {
                unsigned long long lb = 0;
                if (mx) {
                    const uint32_t v = ~static_cast<uint32_t>(mx & 0xffffffffull);
                    const U4 w = philox4x32_10(v >> 2, pos, req, 0u, seed_lo, seed_hi);
                    const uint32_t j = v & 3u;
                    const uint32_t wj = j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w;
                    const float xmax = order_to_float(static_cast<uint32_t>(mx >> 32));   // the logit itself
                    lb = pack_key(__fadd_rn(__fmul_rn(xmax, invT), gumbel_from_word(wj)), v);
                }
                bcast = lb;
                s_best = lb;
            }
            __syncthreads();
            best = bcast;
            // ---- pass 2a: compact the live blocks (block maximum can still reach
            // LB with the largest noise) into a list, in place over bmax; a
            // window of 256 blocks at a time, reads before writes.
            const uint32_t lbo = static_cast<uint32_t>(best >> 32);
            int n_live = 0;
#pragma unroll 1
            for (int w0 = 0; w0 < n_blocks; w0 += kSelThreads) {
                const int blk = w0 + static_cast<int>(threadIdx.x);
                const bool live = blk < n_blocks &&
                                  key_order(__fadd_rn(__fmul_rn(bmax[blk], invT), kNoiseBound)) >= lbo;
                const unsigned bal = __ballot_sync(0xffffffffu, live);
                if (lane == 0) wcount[warp] = __popc(bal);
                __syncthreads();
                int before = n_live, total_w = 0;
#pragma unroll
                for (int i = 0; i < kSelThreads / 32; ++i) {
                    before += i < warp ? wcount[i] : 0;
                    total_w += wcount[i];
                }
                if (live) live_list[before + __popc(bal & ((1u << lane) - 1u))] = blk;
                n_live += total_w;
                __syncthreads();
            }
            // ---- a row with many live blocks goes to the unit kernel: its live
            // list, one unit per chunk that holds live blocks, its state.  (The
            // slot is taken by thread 0 and broadcast; past the scratch's
            // capacity the row is done here.)
            if (hv.cap > 0 && n_live > hv.min_live) {
                if (threadIdx.x == 0) s_heavy = static_cast<int>(atomicAdd(&hv.ctr[0], 1u));
                __syncthreads();
                const int h = s_heavy;
                if (h < hv.cap) {
                    for (int i = static_cast<int>(threadIdx.x); i < n_live; i += kSelThreads)
                        hv.live[static_cast<long long>(h) * n_blocks + i] = static_cast<uint16_t>(live_list[i]);
                    constexpr int bpc = kStreamChunk / kBlock;   // blocks per chunk
                    int n_units = 0;
#pragma unroll 1
                    for (int c0 = 0; c0 < n_chunks; c0 += kSelThreads) {
                        const int c = c0 + static_cast<int>(threadIdx.x);
                        int lo = 0, hi = 0;
                        if (c < n_chunks) {
                            lo = lower_bound_int(live_list, n_live, c * bpc);
                            hi = lower_bound_int(live_list, n_live, (c + 1) * bpc);
                        }
                        const bool has = hi > lo;
                        const unsigned bal = __ballot_sync(0xffffffffu, has);
                        if (lane == 0) wcount[warp] = __popc(bal);
                        __syncthreads();
                        int before = 0, total_w = 0;
#pragma unroll
                        for (int i = 0; i < kSelThreads / 32; ++i) {
                            before += i < warp ? wcount[i] : 0;
                            total_w += wcount[i];
                        }
                        if (threadIdx.x == 0)
                            s_unit0 = static_cast<int>(atomicAdd(&hv.ctr[1], static_cast<unsigned>(total_w)));
                        __syncthreads();
                        if (has) hv.units[s_unit0 + before + __popc(bal & ((1u << lane) - 1u))] = make_int4(h, c, lo, hi);
                        n_units += total_w;
                        __syncthreads();                  // wcount and s_unit0 are reused
                    }
                    if (threadIdx.x == 0) {
                        hv.best[h] = best;
                        hv.row_of[h] = row;
                        hv.remaining[h] = n_units;
                    }
                    __syncthreads();                      // the live list (over bmax) is read
                    continue;                             // the unit kernel writes the token
                }
            }
            // ---- pass 2b: the 4-groups of the live blocks, all threads, kUnroll
            // loads in flight per thread; 32 consecutive items share a block.
            best = groups_pass<kUnroll>(x, 0, n_live * (kBlock / 4), [&](int i) { return live_list[i]; }, V, pos, req,
                                        seed_lo, seed_hi, invT, gtab, g254, best, &s_best);
            best = block_max64(best, red);              // also orders pass 2's reads of bmax before the next row
        }
        if (threadIdx.x == 0)
            tokens[row] = best ? static_cast<int32_t>(~static_cast<uint32_t>(best & 0xffffffffull)) : 0;
    }
    // After a time-out, the copies still in flight (chunks k .. k_issued - 1)
    // land before the CTA's shared memory is released.  The last CTA to leave
    // resets the launch's counters for the next launch that uses them.
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!ok)
            for (long long j = k; j < k_issued; ++j)
                mbar_wait_drain(&fbar[j % kStreamStages], static_cast<uint32_t>((j / kStreamStages) & 1));
        __threadfence();
        if (atomicAdd(&ctr[1], 1u) == gridDim.x - 1) {
            ctr[0] = 0;
            ctr[1] = 0;
            __threadfence();
        }
    }
}

// ------------------------------------------------------------ unit kernel
// The heavy rows' units (see HeavyRows).  Warps 0-7 compute; warp 8 is the
// producer: it draws unit tickets, reads a unit's descriptor, row and live
// blocks into a slot's metadata, copies the unit's chunk into the slot's
// ring buffer (full barrier), and, once the compute warps release the slot
// (empty barrier, one arrival per warp), raises the row's best key with the
// unit's result by a 64-bit atomic maximum -- the unit that brings the row's
// count of units to zero writes its token.  The compute warps run pass 2b
// over the unit's live blocks from shared memory, starting from the row's
// best key when the unit was drawn.  Global latency stays with the producer.
// Exact for the same reason as the streaming kernel: only entries whose bound
// stays below a real key of the row are skipped.
constexpr int kUStages = 3;
constexpr int kUThreads = kSelThreads + 32;

struct UnitMeta {
    int h, c, n_lb, row;
    uint32_t req, pos;
};

size_t unit_smem_bytes() { return static_cast<size_t>(kUStages) * kStreamChunk * 4; }

__global__ void __launch_bounds__(kUThreads, 2)
gumbel_units_kernel(const float* __restrict__ logits, int V, long long ld, const uint32_t* __restrict__ row_req,
                    const int32_t* __restrict__ row_pos, uint32_t seed_lo, uint32_t seed_hi, float invT,
                    int32_t* __restrict__ tokens, const __grid_constant__ NoiseBounds nb, const HeavyRows hv) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float* ring = reinterpret_cast<float*>(smem_raw);    // [kUStages][chunk]
    __shared__ uint64_t full[kUStages], empty[kUStages];
    __shared__ UnitMeta meta[kUStages];                  // h < 0: no more units
    __shared__ int blk[kUStages][kStreamChunk / kBlock];
    __shared__ unsigned long long best0[kUStages];       // the running best of the slot's unit
    __shared__ unsigned long long res[kUStages];         // the slot's unit result, for the producer
    __shared__ unsigned long long red[kUStages][kSelThreads / 32];
    __shared__ float gtab[256];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kUStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kSelThreads / 32);
        }
        fence_mbar_init();
    }
    if (threadIdx.x < 256) gtab[threadIdx.x] = nb.v[threadIdx.x];
    const float g254 = nb.v[254];
    __syncthreads();
    pdl_wait();                                          // the hand-offs of the streaming kernel
    pdl_trigger();
    const int n_blocks = (V + kBlock - 1) / kBlock;
    if (warp == kSelThreads / 32) {
        // ------------------------------------------------ producer warp
        const unsigned n_units = hv.ctr[1];
        long long k = 0;
        bool ok = true;
        auto finish = [&](int s) {                       // lane 0: the unit in slot s is done
            const int h = meta[s].h;
            atomicMax(&hv.best[h], res[s]);
            __threadfence();
            if (atomicSub(&hv.remaining[h], 1) == 1) {   // the row's last unit
                __threadfence();
                const unsigned long long fin = atomicMax(&hv.best[h], 0ull);
                tokens[meta[s].row] = fin ? static_cast<int32_t>(~static_cast<uint32_t>(fin & 0xffffffffull)) : 0;
            }
        };
#pragma unroll 1
        for (;; ++k) {
            const int s = static_cast<int>(k % kUStages);
            if (k >= kUStages) {
                if (!mbar_wait(&empty[s], static_cast<uint32_t>((k / kUStages - 1) & 1), &abort_flag, &g_select_err)) {
                    ok = false;
                    break;
                }
                if (lane == 0) finish(s);
            }
            unsigned t = 0;
            if (lane == 0) t = atomicAdd(&hv.ctr[2], 1u);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t >= n_units) {
                if (lane == 0) {
                    meta[s].h = -1;
                    mbar_arrive(&full[s]);               // the end marker completes the phase
                }
                break;
            }
            const int4 u = hv.units[t];
            const int n_lb = u.w - u.z;
            const int row = hv.row_of[u.x];
            if (lane < n_lb) blk[s][lane] = hv.live[static_cast<long long>(u.x) * n_blocks + u.z + lane];
            if (lane == 0) {
                meta[s] = UnitMeta{u.x, u.y, n_lb, row, row_req[row], static_cast<uint32_t>(row_pos[row]) + 1u};
                best0[s] = *reinterpret_cast<volatile unsigned long long*>(&hv.best[u.x]);
            }
            __syncwarp();
            if (lane == 0) {
                const int n = min(kStreamChunk, V - u.y * kStreamChunk);
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(n) * 4u);
                bulk_g2s(ring + static_cast<long long>(s) * kStreamChunk,
                         logits + static_cast<long long>(row) * ld + static_cast<long long>(u.y) * kStreamChunk,
                         static_cast<uint32_t>(n) * 4u, &full[s]);
            }
        }
        // the units still in the ring when the end marker went in: their results
        if (ok) {
#pragma unroll 1
            for (long long j = k - kUStages + 1; j < k; ++j) {
                if (j < 0) continue;
                const int s = static_cast<int>(j % kUStages);
                if (!mbar_wait(&empty[s], static_cast<uint32_t>((j / kUStages) & 1), &abort_flag, &g_select_err))
                    break;
                if (lane == 0) finish(s);
            }
        }
        // after a time-out, every copy issued lands before the shared memory goes
        if (lane == 0 && *reinterpret_cast<volatile int*>(&abort_flag)) {
            for (int s = 0; s < kUStages; ++s) {
                long long j = k - 1;                     // the last ordinal that used slot s
                while (j >= 0 && j % kUStages != s) --j;
                if (j >= 0) mbar_wait_drain(&full[s], static_cast<uint32_t>((j / kUStages) & 1));
            }
        }
    } else {
        // ------------------------------------------------ compute warps
#pragma unroll 1
        for (long long k = 0;; ++k) {
            const int s = static_cast<int>(k % kUStages);
            if (!mbar_wait(&full[s], static_cast<uint32_t>((k / kUStages) & 1), &abort_flag, &g_select_err)) break;
            const UnitMeta m = meta[s];
            if (m.h < 0) break;
            unsigned long long b = groups_pass<kUnroll>(
                ring + static_cast<long long>(s) * kStreamChunk, static_cast<long long>(m.c) * kStreamChunk,
                m.n_lb * (kBlock / 4), [&](int i) { return blk[s][i]; }, V, m.pos, m.req, seed_lo, seed_hi, invT, gtab,
                g254, best0[s], &best0[s]);
            b = warp_max64(b);
            if (lane == 0) red[s][warp] = b;
            asm volatile("bar.sync 1, %0;" ::"n"(kSelThreads) : "memory");   // the compute warps only
            if (threadIdx.x == 0) {
                unsigned long long r = 0;
#pragma unroll
                for (int w = 0; w < kSelThreads / 32; ++w) r = umax64(r, red[s][w]);
                res[s] = r;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);       // the slot is read (warp 0: and res written)
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------- Gumbel top-k
// [COUPLING]: the Gumbel-max trick gives top-k sampling as it stands -- the k
// largest keys, in decreasing order, are k draws without replacement from
// softmax(x / T) (Kool, van Hoof & Welling, "Stochastic Beams and Where to Find
// Them").  Same keys and order as gumbel_argmax_kernel, so column 0 is its
// token.  One CTA per row: every thread keeps its own k best packed keys
// (sorted, in shared memory); an entry is evaluated exactly only if its bound
// beats the thread's k-th best once the list is full (group bound with the
// largest noise, then the bucket bound of its word); the CTA then takes the
// k largest heads one by one.
constexpr int kTopkThreads = 256;
constexpr int kMaxTopk = 64;

__global__ void __launch_bounds__(kTopkThreads)
gumbel_topk_kernel(const float* __restrict__ logits, int V, long long ld, const uint32_t* __restrict__ row_req,
                   const int32_t* __restrict__ row_pos, uint32_t seed_lo, uint32_t seed_hi, float invT, int greedy,
                   int k, int32_t* __restrict__ out) {
    extern __shared__ __align__(16) unsigned long long lists[];   // [k][kTopkThreads]
    __shared__ float tab[256];                                   // largest noise of each top-byte bucket
    __shared__ unsigned long long red[kTopkThreads / 32];
    const int t = threadIdx.x;
    tab[t] = gumbel_from_word((static_cast<uint32_t>(t) << 24) | 0x00ffffffu);
    for (int i = 0; i < k; ++i) lists[i * kTopkThreads + t] = 0ull;
    __syncthreads();
    pdl_wait();
    pdl_trigger();
    const long long row = blockIdx.x;
    const float* x = logits + row * ld;
    const uint32_t req = row_req[row];
    const uint32_t pos = static_cast<uint32_t>(row_pos[row]) + 1u;
    const float gmax = tab[255];
    int count = 0;
    unsigned long long kth = 0;          // the thread's k-th best once its list is full
    auto insert = [&](unsigned long long pk) {
        int i = count < k ? count : k - 1;
        while (i > 0 && lists[(i - 1) * kTopkThreads + t] < pk) {
            lists[i * kTopkThreads + t] = lists[(i - 1) * kTopkThreads + t];
            --i;
        }
        lists[i * kTopkThreads + t] = pk;
        if (count < k) ++count;
        if (count == k) kth = lists[(k - 1) * kTopkThreads + t];
    };
    for (int gi = t; gi < V / 4; gi += kTopkThreads) {
        const float4 v4 = *reinterpret_cast<const float4*>(x + 4 * gi);
        const float e[4] = {v4.x, v4.y, v4.z, v4.w};
        const uint32_t v0 = static_cast<uint32_t>(4 * gi);
        if (greedy) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const unsigned long long pk = pack_key(e[j], v0 + j);
                if (pk > kth) insert(pk);
            }
            continue;
        }
        const float m4 = fmaxf(fmaxf(e[0], e[1]), fmaxf(e[2], e[3]));
        const unsigned long long gb =
            (static_cast<unsigned long long>(key_order(__fadd_rn(__fmul_rn(m4, invT), gmax))) << 32) |
            static_cast<unsigned long long>(~v0);
        if (count == k && gb <= kth) continue;
        const U4 w = philox4x32_10(v0 >> 2, pos, req, 0u, seed_lo, seed_hi);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = __fmul_rn(e[j], invT);
            const unsigned long long eb =
                (static_cast<unsigned long long>(key_order(__fadd_rn(a, tab[ws[j] >> 24]))) << 32) |
                static_cast<unsigned long long>(~(v0 + j));
            if (count == k && eb <= kth) continue;
            const unsigned long long pk = pack_key(__fadd_rn(a, gumbel_from_word(ws[j])), v0 + j);
            if (pk > kth) insert(pk);
        }
    }
    // Merge: k rounds of the largest head.
    int head = 0;
    for (int i = 0; i < k; ++i) {
        const unsigned long long mine = head < count ? lists[head * kTopkThreads + t] : 0ull;
        const unsigned long long best = block_max64(mine, red);
        if (best != 0 && mine == best) ++head;
        if (t == 0) out[row * k + i] = best ? static_cast<int32_t>(~static_cast<uint32_t>(best & 0xffffffffull)) : -1;
    }
}

__global__ void gumbel_noise_kernel(uint32_t seed_lo, uint32_t seed_hi, const uint32_t* __restrict__ row_req,
                                    const int32_t* __restrict__ row_pos, int V, float* __restrict__ g) {
    pdl_wait();
    pdl_trigger();
    const long long row = blockIdx.y;
    const uint32_t req = row_req[row];
    const uint32_t pos = static_cast<uint32_t>(row_pos[row]) + 1u;
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
        const U4 w = philox4x32_10(static_cast<uint32_t>(v) >> 2, pos, req, 0u, seed_lo, seed_hi);
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
        g[row * V + v] = gumbel_from_word(words[v & 3]);
    }
}

__global__ void gumbel_words_kernel(const uint32_t* __restrict__ words, long long n, float* __restrict__ g) {
    pdl_wait();
    pdl_trigger();
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        g[i] = gumbel_from_word(words[i]);
}

// One thread per request: first mismatch of target vs draft.
__global__ void verify_accept_kernel(const int32_t* __restrict__ target, const int32_t* __restrict__ draft,
                                     const int32_t* __restrict__ p0, int N, int K,
                                     int32_t* __restrict__ accept_len, int32_t* __restrict__ new_len) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= N) return;
    int L = K;
    for (int j = 0; j < K; ++j) {
        if (target[static_cast<long long>(r) * K + j] != draft[static_cast<long long>(r) * K + j]) {
            L = j + 1;
            break;
        }
    }
    accept_len[r] = L;
    new_len[r] = p0[r] + L;
}


// A row is heavy when more than a quarter of its blocks (and more than 32)
// stay live: a unit streams a whole chunk, which pays off only where most of
// its blocks are live (a peaked row keeps a few live blocks and stays).  At
// most an eighth of the rows are handed off: when most rows are flat every
// CTA has Philox work anyway, and a row re-read right after its pass 1 still
// sits in L2.
constexpr int kHeavyMinLive = 32;

size_t align16(size_t n) { return (n + 15) & ~static_cast<size_t>(15); }

// The heavy-row scratch of a call with R rows of V logits, carved from the
// caller's workspace: {counters}{best}{row_of}{remaining}{units}{live} for up
// to R / 8 rows (at least one).
struct HeavyLayout {
    int cap, n_blocks, n_chunks;
    size_t o_best, o_row, o_rem, o_units, o_live, bytes;
};

HeavyLayout heavy_layout(int R, int V) {
    HeavyLayout L;
    L.cap = std::max(1, R / 8);
    L.n_blocks = (V + kBlock - 1) / kBlock;
    L.n_chunks = (V + kStreamChunk - 1) / kStreamChunk;
    L.o_best = 64;
    L.o_row = L.o_best + align16(static_cast<size_t>(L.cap) * 8);
    L.o_rem = L.o_row + align16(static_cast<size_t>(L.cap) * 4);
    L.o_units = L.o_rem + align16(static_cast<size_t>(L.cap) * 4);
    L.o_live = L.o_units + static_cast<size_t>(L.cap) * L.n_chunks * 16;
    L.bytes = L.o_live + align16(static_cast<size_t>(L.cap) * L.n_blocks * 2);
    return L;
}

// Persistent launch of the streaming kernel: as many CTAs as fit on the GPU,
// at most one per row; CTA b takes rows b, b + grid, ...  With a workspace
// and T > 0, flat rows are handed to the unit kernel, launched right after
// (the workspace's counters are cleared first, in stream order).
int launch_stream_select(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                         const int32_t* row_pos, uint64_t seed, float invT, int greedy, int32_t* tokens,
                         void* workspace, cudaStream_t stream) {
    const size_t smem = stream_smem_bytes(V);
    const size_t unit_smem = unit_smem_bytes();
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_status(de);
    if (dev < 0 || dev >= kMaxDevices) return BIV_ERR_DEVICE;
    int per_sm = 0, unit_per_sm = 0;
    unsigned int* ctr_base = nullptr;
    {
        // per device, from any host thread: the kernel attributes, the counter
        // ring's device address and the occupancy at this shared-memory size
        static std::mutex mu;
        static unsigned int* ctr_dev[kMaxDevices] = {};
        static int unit_occ[kMaxDevices] = {};
        static size_t occ_smem[kMaxDevices] = {};
        static int occ_per_sm[kMaxDevices] = {};
        std::lock_guard<std::mutex> lock(mu);
        if (!ctr_dev[dev]) {
            cudaError_t e = cudaFuncSetAttribute(gumbel_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(stream_smem_bytes(kMaxStreamV)));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gumbel_units_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(unit_smem));
            int n = 0;
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gumbel_units_kernel, kUThreads, unit_smem);
            if (e != cudaSuccess) return cuda_status(e);
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_stream_ctr);
            if (e != cudaSuccess) return cuda_status(e);
            unit_occ[dev] = std::max(1, n);
            ctr_dev[dev] = static_cast<unsigned int*>(p);
        }
        unit_per_sm = unit_occ[dev];
        if (occ_smem[dev] != smem) {
            int n = 0;
            cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gumbel_stream_kernel, kSelThreads, smem);
            if (e != cudaSuccess) return cuda_status(e);
            occ_smem[dev] = smem;
            occ_per_sm[dev] = std::max(1, n);
        }
        per_sm = occ_per_sm[dev];
        ctr_base = ctr_dev[dev];
    }
    // Each launch takes the next counter pair of the ring (launches in flight
    // at the same time on different streams must not share one).
    static std::atomic<unsigned> next_slot{0};
    unsigned int* ctr = ctr_base + 2 * (next_slot.fetch_add(1u) % kCtrSlots);
    const long long cap = static_cast<long long>(num_sms()) * per_sm;
    const int grid = static_cast<int>(std::min<long long>(R, cap));
    const uint32_t seed_lo = static_cast<uint32_t>(seed & 0xffffffffull), seed_hi = static_cast<uint32_t>(seed >> 32);

    HeavyRows hv = {};
    const bool hand_off = workspace != nullptr && !greedy;
    if (hand_off) {
        const HeavyLayout L = heavy_layout(R, V);
        uint8_t* b = static_cast<uint8_t*>(workspace);
        const cudaError_t e = cudaMemsetAsync(b, 0, 64, stream);   // the counters
        if (e != cudaSuccess) return cuda_status(e);
        hv.ctr = reinterpret_cast<unsigned int*>(b);
        hv.best = reinterpret_cast<unsigned long long*>(b + L.o_best);
        hv.row_of = reinterpret_cast<int*>(b + L.o_row);
        hv.remaining = reinterpret_cast<int*>(b + L.o_rem);
        hv.units = reinterpret_cast<int4*>(b + L.o_units);
        hv.live = reinterpret_cast<uint16_t*>(b + L.o_live);
        hv.cap = L.cap;
        hv.min_live = std::max(kHeavyMinLive, L.n_blocks / 4);
    }
    int st = launch_pdl(gumbel_stream_kernel, dim3(static_cast<unsigned>(grid)), dim3(kSelThreads), smem, stream,
                        logits, R, V, ld, row_req, row_pos, seed_lo, seed_hi, invT, greedy, tokens, ctr,
                        noise_bounds(), hv);
    if (st == BIV_OK && hand_off) {
        const int ugrid = static_cast<int>(std::min<long long>(
            static_cast<long long>(hv.cap) * ((V + kStreamChunk - 1) / kStreamChunk),
            static_cast<long long>(num_sms()) * unit_per_sm));
        st = launch_pdl(gumbel_units_kernel, dim3(static_cast<unsigned>(ugrid)), dim3(kUThreads), unit_smem,
                        stream, logits, V, ld, row_req, row_pos, seed_lo, seed_hi, invT, tokens, noise_bounds(), hv);
    }
    return st;
}

}  // namespace
}  // namespace biv

using namespace biv;

// Both selection entry points; workspace (or null) as biv_gumbel_argmax_ws.
static int gumbel_argmax_impl(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                              const int32_t* row_pos, uint64_t seed, float temperature, int32_t* tokens,
                              void* workspace, biv_stream_t stream) {
    if (R < 0 || V < 4 || ld < V) return BIV_ERR_SHAPE;
    if (V % 4 != 0 || ld % 4 != 0) return BIV_ERR_SHAPE;
    if (!(temperature >= 0.0f) || !(temperature < INFINITY)) return BIV_ERR_VALUE;
    if (R == 0) return BIV_OK;
    if (!logits || !row_req || !row_pos || !tokens) return BIV_ERR_NULL;
    if (!aligned16(logits)) return BIV_ERR_ALIGN;
    const int slice = ((V / 4 + kClusterSize - 1) / kClusterSize) * 4;
    if (V > kMaxStreamV) return BIV_ERR_UNSUPPORTED;
    const int greedy = temperature == 0.0f;
    const float invT = greedy ? 0.0f : 1.0f / temperature;   // fl(1/T), IEEE division on the host
    // Many rows (two or more per SM) or a row too wide for one cluster: a CTA
    // streams whole rows.  Few rows: a cluster of eight CTAs shares each row.
    if (R >= 2 * num_sms() || slice > kMaxSliceFloats) {
        return launch_stream_select(logits, R, V, ld, row_req, row_pos, seed, invT, greedy, tokens, workspace,
                                    reinterpret_cast<cudaStream_t>(stream));
    }
    if (static_cast<long long>(R) * kClusterSize > 0x7fffffffLL) return BIV_ERR_SHAPE;
    const size_t smem = static_cast<size_t>(slice) * 5;

    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_status(de);
    static DeviceOnce once;
    const int st = once.run(dev, [] {
        return cuda_status(cudaFuncSetAttribute(gumbel_argmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(kMaxSliceFloats * 5)));
    });
    if (st != BIV_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(R) * kClusterSize, 1, 1);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterSize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gumbel_argmax_kernel, logits, V, ld, slice, row_req, row_pos,
                                       static_cast<uint32_t>(seed & 0xffffffffull),
                                       static_cast<uint32_t>(seed >> 32), invT, greedy, tokens, noise_bounds());
    if (e != cudaSuccess) return cuda_status(e);
    return launch_status();
}

extern "C" int biv_gumbel_argmax(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                                 const int32_t* row_pos, uint64_t seed, float temperature, int32_t* tokens,
                                 biv_stream_t stream) {
    BIV_TRACE_CALL();
    return gumbel_argmax_impl(logits, R, V, ld, row_req, row_pos, seed, temperature, tokens, nullptr, stream);
}

extern "C" size_t biv_gumbel_argmax_workspace_size(int R, int V) {
    if (R <= 0 || V < 4 || V % 4 != 0 || V > kMaxStreamV) return 0;
    return heavy_layout(R, V).bytes;
}

extern "C" int biv_gumbel_argmax_ws(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                                    const int32_t* row_pos, uint64_t seed, float temperature, int32_t* tokens,
                                    void* workspace, size_t ws_bytes, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (R < 0 || V < 4 || ld < V || V % 4 != 0 || ld % 4 != 0) return BIV_ERR_SHAPE;
    if (R > 0) {
        if (!workspace) return BIV_ERR_NULL;
        if (!aligned16(workspace)) return BIV_ERR_ALIGN;
        if (ws_bytes < biv_gumbel_argmax_workspace_size(R, V)) return BIV_ERR_SHAPE;
    }
    return gumbel_argmax_impl(logits, R, V, ld, row_req, row_pos, seed, temperature, tokens, workspace, stream);
}

extern "C" int biv_gumbel_topk(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                               const int32_t* row_pos, uint64_t seed, float temperature, int k, int32_t* out,
                               biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (R < 0 || V < 4 || ld < V || V % 4 != 0 || ld % 4 != 0) return BIV_ERR_SHAPE;
    if (k < 1 || k > kMaxTopk || k > V) return BIV_ERR_SHAPE;
    if (!(temperature >= 0.0f) || !(temperature < INFINITY)) return BIV_ERR_VALUE;
    if (R == 0) return BIV_OK;
    if (!logits || !row_req || !row_pos || !out) return BIV_ERR_NULL;
    if (!aligned16(logits)) return BIV_ERR_ALIGN;
    const int greedy = temperature == 0.0f;
    const float invT = greedy ? 0.0f : 1.0f / temperature;   // fl(1/T), IEEE division on the host
    const size_t smem = static_cast<size_t>(k) * kTopkThreads * sizeof(unsigned long long);
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_status(de);
    static DeviceOnce once;
    const int st = once.run(dev, [] {
        return cuda_status(cudaFuncSetAttribute(gumbel_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                static_cast<int>(kMaxTopk * kTopkThreads * sizeof(unsigned long long))));
    });
    if (st != BIV_OK) return st;
    return launch_pdl(gumbel_topk_kernel, dim3(static_cast<unsigned>(R)), dim3(kTopkThreads), smem,
                      reinterpret_cast<cudaStream_t>(stream), logits, V, ld, row_req, row_pos,
                      static_cast<uint32_t>(seed & 0xffffffffull), static_cast<uint32_t>(seed >> 32), invT, greedy, k,
                      out);
}

extern "C" int biv_gumbel_noise(uint64_t seed, const uint32_t* row_req, const int32_t* row_pos, int R, int V,
                                float* g, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (R < 0 || V < 0 || R > 65535) return BIV_ERR_SHAPE;
    if (R == 0 || V == 0) return BIV_OK;
    if (!row_req || !row_pos || !g) return BIV_ERR_NULL;
    const int blocks = std::min((V + 255) / 256, 1024);
    return launch_pdl(gumbel_noise_kernel, dim3(blocks, R), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<uint32_t>(seed & 0xffffffffull), static_cast<uint32_t>(seed >> 32), row_req,
                      row_pos, V, g);
}

extern "C" int biv_gumbel_from_words(const uint32_t* words, long long n, float* g, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (n < 0) return BIV_ERR_SHAPE;
    if (n == 0) return BIV_OK;
    if (!words || !g) return BIV_ERR_NULL;
    const long long blocks = std::min<long long>((n + 255) / 256, 4096);
    return launch_pdl(gumbel_words_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                      reinterpret_cast<cudaStream_t>(stream), words, n, g);
}

extern "C" int biv_verify_accept(const int32_t* target, const int32_t* draft, const int32_t* p0, int N, int K,
                                 int32_t* accept_len, int32_t* new_len, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (N < 0 || K < 1) return BIV_ERR_SHAPE;
    if (N == 0) return BIV_OK;
    if (!target || !draft || !p0 || !accept_len || !new_len) return BIV_ERR_NULL;
    return launch_pdl(verify_accept_kernel, dim3((N + 127) / 128), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      target, draft, p0, N, K, accept_len, new_len);
}

extern "C" int biv_gumbel_bucket_bounds(float* bounds_out) {
    BIV_TRACE_CALL();
    if (!bounds_out) return BIV_ERR_NULL;
    const NoiseBounds& nb = noise_bounds();
    for (int b = 0; b < 256; ++b) bounds_out[b] = nb.v[b];
    return BIV_OK;
}
