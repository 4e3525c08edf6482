// Fixed-split decode attention, RoPE and the verifier's KV overwrite.
//
// [DVR] para 1: batch-invariant attention uses a fixed KV-split size with no
// adaptation to sequence length or GPU load.  [DVR] para 3: the verifier
// overwrites the fast path's cache rows with its own values before they are
// attended to.  [GUIDE] GQA tile rule: the G query heads that share a KV head,
// times the verified rows of one request, fill one 128-row MMA tile
// (G * (1 + D) <= 128).
//
// Phase 1 (attn_tc_kernel): a work item is (row tile, KV head, split of 256
// absolute positions); the tile holds up to 128/G consecutive rows of one
// request times its G query heads, so K and V of the split are read once for
// all of them.  S = Q K^T and O = P V run on the tensor cores with the
// accumulators in TMEM; the softmax over the whole split runs between them
// in registers, masking keys past each row's own position with a select.
// The split's partial (max, sum, unnormalised output) goes to the caller's
// workspace.  Phase 2 (attn_combine_kernel) combines the splits 0..p/256 of
// each (row, head) in increasing order.  Nothing in a row's arithmetic
// depends on the other rows of the tile or the batch: masked keys contribute
// exact zeros, the MMAs contract in fixed 16-wide steps and every sum has a
// fixed order.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_attn_err)

constexpr int HD = BIV_HEAD_DIM;        // 128
constexpr int SPLIT = BIV_KV_SPLIT;     // 256
constexpr int ROWB = HD * 2;            // 256 bytes per K/V row
constexpr int ATTN_THREADS = 256;

BIV_DEV void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
BIV_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
BIV_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct AttnParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* kc;
    const __nv_bfloat16* vc;
    const int32_t* row_slot;
    const int32_t* row_pos;
    float* ws_o;      // [W][Hq][S_max][HD]
    float* ws_m;      // [W][Hq][S_max]
    float* ws_l;      // [W][Hq][S_max]
    int W, rows_per_group, tile_rows, tiles_per_group, n_tiles;
    int Hq, Hkv, G, n_slots, max_len, s_max;
    float scale_log2;  // log2(e) / sqrt(HD)
};

// Is row w usable for a tile whose first row is w0 (device-side checks)?
BIV_DEV bool row_ok(const AttnParams& P, int w, int slot0) {
    const int s = P.row_slot[w], p = P.row_pos[w];
    if (s < 0 || s >= P.n_slots || p < 0 || p >= P.max_len) {
        atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
        return false;
    }
    if (s != slot0) {
        atomicOr(&g_attn_err, BIV_DEVERR_GROUP);
        return false;
    }
    return true;
}

// First row and row count of tile t (row-major groups of rows_per_group rows,
// each cut into tiles of tile_rows).
BIV_DEV void tile_rows_of(const AttnParams& P, int t, int& row0, int& nr) {
    const int group = t / P.tiles_per_group;
    const int sub = t - group * P.tiles_per_group;
    row0 = group * P.rows_per_group + sub * P.tile_rows;
    const int row_end = min(min(row0 + P.tile_rows, (group + 1) * P.rows_per_group), P.W);
    nr = row_end - row0;
}

// Largest position of a usable row of tile t (-1 if none).  A tile whose
// first row's slot is out of range raises BIV_DEVERR_INDEX here (it is never
// processed); the other row errors are raised where the tile is processed.
BIV_DEV int tile_maxpos(const AttnParams& P, int t) {
    int row0, nr;
    tile_rows_of(P, t, row0, nr);
    if (nr <= 0) return -1;
    const int slot0 = P.row_slot[row0];
    if (slot0 < 0 || slot0 >= P.n_slots) {
        atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
        return -1;
    }
    int m = -1;
    for (int w = row0; w < row0 + nr; ++w) {
        const int s = P.row_slot[w], p = P.row_pos[w];
        if (s == slot0 && p >= 0 && p < P.max_len) m = max(m, p);
    }
    return m;
}

constexpr int kMaxTilesSmem = 2048;
constexpr int kMaxRowsSmem = 2048;                 // rows whose usable positions are tabulated

// Per-tile tables in shared memory, built by all threads of the CTA: the
// largest usable position of each tile (-1: none), its first row's cache
// slot, and the exclusive prefix sums of its live work items
// (Hkv * (tmax / SPLIT + 1) each); s_pref[tile_cap] is the live total.
// Returns whether the tables cover every tile (else callers fall back to all
// (split, KV head, tile) triples with the dead ones skipped).
// Only the first ATTN_THREADS threads of the CTA fill the tables; every
// thread of the CTA must call this (it contains the CTA barriers).
BIV_DEV bool build_tile_tables(const AttnParams& P, int* s_tmax, int* s_pref, int* s_slot0, int* s_wsum,
                               int* s_rpos, int* s_gmin, int tile_cap = kMaxTilesSmem, int row_cap = kMaxRowsSmem) {
    const int n_tiles = P.n_tiles;
    const bool act = threadIdx.x < ATTN_THREADS;
    // s_rpos: each row's usable position (-1: none), when every row is tabulated
    const bool rows_tab = P.W <= row_cap && n_tiles <= tile_cap;
    // Largest usable position of each tile, one thread per row (independent
    // loads); tiles past the table are scanned where they are processed.
    for (int t = threadIdx.x; act && t < min(n_tiles, tile_cap); t += ATTN_THREADS) {
        s_tmax[t] = -1;
        s_gmin[t] = 0x7fffffff;             // per row group (there are no more groups than tiles)
    }
    __syncthreads();
    for (int w = threadIdx.x; act && w < P.W; w += ATTN_THREADS) {
        const int group = w / P.rows_per_group;
        const int sub = (w - group * P.rows_per_group) / P.tile_rows;
        const int t = group * P.tiles_per_group + sub;
        if (t >= tile_cap) break;                            // rows only grow the tile index
        const int row0 = group * P.rows_per_group + sub * P.tile_rows;
        // the three loads are independent: one round trip (the inputs are cold
        // in HBM when the kernel starts)
        const int slot0 = P.row_slot[row0];
        const int s = P.row_slot[w], p = P.row_pos[w];
        if (w == row0) s_slot0[t] = slot0;
        if (slot0 < 0 || slot0 >= P.n_slots) {
            if (w == row0 && blockIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
            if (rows_tab) s_rpos[w] = -1;
            continue;
        }
        // the row checks of row_ok(), raised once (by CTA 0)
        int vp = -1;
        if (s < 0 || s >= P.n_slots || p < 0 || p >= P.max_len) {
            if (blockIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
        } else if (s != slot0) {
            if (blockIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_GROUP);
        } else {
            vp = p;
            atomicMax(&s_tmax[t], p);
            atomicMin(&s_gmin[group], p);
        }
        if (rows_tab) s_rpos[w] = vp;
    }
    __syncthreads();
    // Live work items: tile t has Hkv * (s_tmax[t] / SPLIT + 1) of them (none
    // if no row is usable); s_pref holds their exclusive prefix sums, so the
    // CTAs can deal out exactly the live items, consecutive ones to
    // consecutive CTAs.  Tables too large for shared memory fall back to all
    // (split, KV head, tile) triples with the dead ones skipped.
    const bool live_mode = n_tiles <= tile_cap;
    if (live_mode) {
        // thread i scans tiles [i * per, (i + 1) * per); warp and block prefix
        const int per = (n_tiles + ATTN_THREADS - 1) / ATTN_THREADS;
        const int t0 = act ? min(static_cast<int>(threadIdx.x) * per, n_tiles) : n_tiles;
        const int t1 = min(t0 + per, n_tiles);
        int sum = 0;
        for (int t = t0; t < t1; ++t) sum += s_tmax[t] >= 0 ? P.Hkv * (s_tmax[t] / SPLIT + 1) : 0;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int inc = sum;                                       // inclusive scan over the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31 && act) s_wsum[warp] = inc;
        __syncthreads();
        int base = inc - sum;
        for (int w = 0; act && w < warp; ++w) base += s_wsum[w];
        for (int t = t0; t < t1; ++t) {
            s_pref[t] = base;
            base += s_tmax[t] >= 0 ? P.Hkv * (s_tmax[t] / SPLIT + 1) : 0;
        }
        if (threadIdx.x == ATTN_THREADS - 1) s_pref[tile_cap] = base;        // the live total
        __syncthreads();
    }
    return live_mode;
}

// ------------------------------------------------- tensor-core split kernel
// Phase 1 on the 5th-generation tensor cores.  A work item is (row tile, KV
// head, split of 256 absolute positions); persistent CTAs deal out the live
// items (build_tile_tables).  Per item, with M = 64 or 128 MMA rows:
//   S = Q K^T   tcgen05.mma M x 128 x 16, 8 k-steps per 128-key half, fp32
//               accumulators in TMEM columns [0, 256)
//   softmax     the 8 warps read S rows from TMEM, scale them into log2
//               units, mask keys past each row's own position with a select,
//               take the row maximum m over the whole split, p = 2^(s - m),
//               the fp32 sum l of p, and store bf16 p into shared memory as
//               the A operand of
//   O = P V     tcgen05.mma M x 128 x 16 over the split's 16-key steps (V is
//               the MN-major B operand: one row of dims per key), fp32 in
//               TMEM columns [256, 384)
//   partial     (m, l, O) of every tile row that reaches the split, to the
//               workspace that attn_combine_kernel reads.
// Both products contract in whole 16-wide steps in a fixed order and every
// row's arithmetic touches only its own S / P / O row, so a row's result does
// not depend on the rest of the tile or the batch.  K and V of a split arrive
// as 128-key TMA boxes ([2 dim halves][128 keys][128 B], 128-byte swizzle).
// Loads run ahead: the next item's K (M = 64) and Q as soon as this item's S
// is in TMEM, its V (and K for M = 128, whose P reuses K's space) as soon as
// P V is.
constexpr int kTcKeyHalfBytes = 2 * 128 * 128;    // one 128-key box of K or V: 32 KiB
constexpr uint32_t kTmemCols = 512;                // S: [0, 256), O: [256, 384)

template <int M>
constexpr size_t tc_smem_bytes() {
    return 1024 + static_cast<size_t>(M) * 256 + 4 * kTcKeyHalfBytes + (M == 64 ? M * 512 : 0);
}

// MN-major shared-memory descriptor for V with 128-byte swizzle: 64 dims
// (128 B) per swizzled row, one row per key; 8-key atoms 1 KiB apart (stride
// offset), the two 64-dim halves of a box `half_stride` bytes apart (leading
// offset; 16 KiB for a 128-key box) -- the reading a layout probe confirmed
// on the GB300.
BIV_DEV uint64_t sw128_mnmajor_desc(uint32_t smem_addr, uint32_t half_stride = 16384u) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(half_stride >> 4) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

struct TcItem {
    int tile, kvh, split, maxpos, slot0;
};

// Work item `item` in the live (or, past the tables, dense) numbering.
BIV_DEV TcItem tc_decode(const AttnParams& P, bool live_mode, long long item, const int* s_pref,
                         const int* s_tmax, const int* s_slot0) {
    TcItem it;
    if (live_mode) {
        int lo = 0, hi = P.n_tiles - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pref[mid] <= item) lo = mid; else hi = mid - 1;
        }
        it.tile = lo;
        const int r = static_cast<int>(item - s_pref[lo]);
        it.kvh = r % P.Hkv;
        it.split = r / P.Hkv;
        it.maxpos = s_tmax[lo];
        it.slot0 = s_slot0[lo];
    } else {
        it.tile = static_cast<int>(item % P.n_tiles);
        const long long rest = item / P.n_tiles;
        it.kvh = static_cast<int>(rest % P.Hkv);
        it.split = static_cast<int>(rest / P.Hkv);
        it.maxpos = tile_maxpos(P, it.tile);
        int row0, nr;
        tile_rows_of(P, it.tile, row0, nr);
        it.slot0 = nr > 0 ? P.row_slot[row0] : -1;
    }
    return it;
}

// Largest of the first min(lim + 1, N) raw scores v[0 ..] (-inf if none): a
// maximum is exact in any order, so four interleaved partial maxima are used.
template <int N>
BIV_DEV float masked_max(const uint32_t* v, int lim) {
    float a[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (lim >= N - 1) {
#pragma unroll
        for (int t = 0; t < N; ++t) a[t & 3] = fmaxf(a[t & 3], __uint_as_float(v[t]));
    } else {
#pragma unroll
        for (int t = 0; t < N; ++t)
            if (t <= lim) a[t & 3] = fmaxf(a[t & 3], __uint_as_float(v[t]));
    }
    return fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
}

// One 16-key group of a row: p_t = 2^(s_t sl2 - m) (one fused multiply-add
// and the hardware base-2 exponential), 0 for keys t > lim; the p_t as bf16
// pairs into pk[0..7]; returns their fp32 sum taken in key order.
BIV_DEV float softmax_group(const uint32_t* v, float sl2, float nmu, int lim, uint32_t* pk) {
    float p[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) p[t] = ex2_approx(fmaf(__uint_as_float(v[t]), sl2, nmu));
    if (lim < 15) {
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t > lim) p[t] = 0.0f;
    }
    float lg = 0.0f;
#pragma unroll
    for (int t = 0; t < 16; ++t) lg += p[t];
#pragma unroll
    for (int t = 0; t < 8; ++t) pk[t] = pack_bf16x2(p[2 * t], p[2 * t + 1]);
    return lg;
}

template <int M>
__global__ void __launch_bounds__(ATTN_THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmK2, const __grid_constant__ CUtensorMap tmV2,
               const AttnParams P) {
    static_assert(M == 64 || M == 128, "MMA rows");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                                // [2 dim halves][M rows][128 B]
    uint8_t* sK = sQ + M * 256;                        // [2 key halves][2 dim halves][128 keys][128 B]
    uint8_t* sV = sK + 2 * kTcKeyHalfBytes;
    uint8_t* sP = M == 64 ? sV + 2 * kTcKeyHalfBytes : sK;   // [4 key quarters][M rows][128 B]
    const uint32_t uQ = smem_u32(sQ), uK = smem_u32(sK), uV = smem_u32(sV), uP = smem_u32(sP);

    __shared__ int s_pos[BIV_ATTN_TILE];
    __shared__ __align__(8) uint64_t kbar[2], vbar[2], sbar, obar;
    __shared__ uint32_t s_tmem;
    __shared__ int abort_flag;
    __shared__ float s_mx[2][128], s_sum[2][128], s_rowm[128];
    __shared__ int s_tmax[kMaxTilesSmem];
    __shared__ int s_pref[kMaxTilesSmem + 1];
    __shared__ int s_slot0[kMaxTilesSmem];
    __shared__ int s_wsum[ATTN_THREADS / 32];
    __shared__ int s_rpos[kMaxRowsSmem];
    __shared__ int s_gmin[kMaxTilesSmem];                      // smallest usable position of each row group

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kbar[i], 1);
            mbar_init(&vbar[i], 1);
        }
        mbar_init(&sbar, 1);
        mbar_init(&obar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmK2);
        prefetch_tensormap(&tmV2);
    }
    tc_fence_before();
    // The tile tables read only the window's slots and positions, inputs of
    // the call rather than outputs of the previous kernel: built while that
    // kernel finishes.  Q, K and V are read after the wait.
    const bool live_mode = build_tile_tables(P, s_tmax, s_pref, s_slot0, s_wsum, s_rpos, s_gmin);   // ends with a barrier
    const bool rows_tab = P.W <= kMaxRowsSmem && P.n_tiles <= kMaxTilesSmem;
    tc_fence_after();
    uint32_t early = 0;                              // thread 0: key halves of the first item already requested
    const uint32_t tS = s_tmem, tO = s_tmem + 256;
    const long long n_work =
        live_mode ? s_pref[kMaxTilesSmem] : static_cast<long long>(P.s_max) * P.Hkv * P.n_tiles;

    // Barrier phases: *_use counts the phases every thread has waited for (the
    // next wait targets parity use & 1); thread 0 also counts the phases it
    // has started (*_iss) and seen complete (*_seen), to drain after a time-out.
    uint32_t k_use[2] = {0u, 0u}, v_use[2] = {0u, 0u}, s_use = 0u, o_use = 0u;
    uint32_t k_iss[2] = {0u, 0u}, v_iss[2] = {0u, 0u}, s_iss = 0u, o_iss = 0u;
    uint32_t k_seen[2] = {0u, 0u}, v_seen[2] = {0u, 0u}, s_seen = 0u, o_seen = 0u;

    auto n_keys_of = [&](const TcItem& it) { return min(SPLIT, it.maxpos + 1 - it.split * SPLIT); };
    // thread 0: the K or V of an item as one box ([2 dim halves][R keys][128 B],
    // R = 256 for a split with more than 128 keys, else 128), on bars[0]
    auto load_kv = [&](const CUtensorMap* map, const CUtensorMap* map2, uint8_t* dst, uint64_t* bars, uint32_t* iss,
                       const TcItem& it) {
        const int nkh = n_keys_of(it) > 128 ? 2 : 1;
        const int kv_row = (it.slot0 * P.Hkv + it.kvh) * P.max_len + it.split * SPLIT;
        mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(nkh * kTcKeyHalfBytes));
        tma_load_3d(dst, nkh == 2 ? map2 : map, &bars[0], 0, kv_row, 0, policy_evict_first());
        ++iss[0];
    };
    // all threads: the item's Q rows into sQ (K-major, 128-byte swizzle)
    // Thread x copies 16-byte piece c = x % 16 of tile rows t = x / 16 + 16 j:
    // the piece and the row's swizzle phase (t & 7) are the same for every j,
    // and (i, g) = (t / G, t % G) advance by fixed steps, so the loop has no
    // division.
    const int q_c = threadIdx.x & 15, q_t0 = threadIdx.x >> 4;
    const uint32_t q_dst0 = uQ + (q_c >> 3) * (M * 128) + q_t0 * 128 + (((q_c & 7) ^ (q_t0 & 7)) << 4);
    const int q_di = 16 / P.G, q_dg = 16 % P.G;
    const int q_i0 = q_t0 / P.G, q_g0 = q_t0 % P.G;
    auto load_q = [&](const TcItem& it) {
        int row0, nr;
        tile_rows_of(P, it.tile, row0, nr);
        const int T = nr * P.G;
        const __nv_bfloat16* base = P.q + (static_cast<long long>(row0) * P.Hq + it.kvh * P.G) * HD + q_c * 8;
        int i = q_i0, g = q_g0;
        for (int t = q_t0, j = 0; t < T; t += 16, ++j) {
            cp_async16(q_dst0 + static_cast<uint32_t>(j) * 2048u, base + (static_cast<long long>(i) * P.Hq + g) * HD);
            i += q_di;
            g += q_dg;
            if (g >= P.G) {
                g -= P.G;
                ++i;
            }
        }
        cp_async_commit();
    };
    // the CTA's next item at or after `from` that has work (dense numbering skips dead ones)
    auto next_live = [&](long long from) {
        for (long long j = from; j < n_work; j += gridDim.x) {
            if (live_mode) return j;
            const TcItem it = tc_decode(P, false, j, s_pref, s_tmax, s_slot0);
            if (it.maxpos >= it.split * SPLIT) return j;
        }
        return n_work;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&abort_flag) != 0; };
    // thread 0: wait for the next phase of a load barrier before issuing MMAs
    auto take = [&](uint64_t* bar, uint32_t use, uint32_t& seen) {
        const bool got = mbar_wait(bar, use & 1u, &abort_flag, &g_attn_err, true);
        if (got) ++seen;
        return got;
    };

    long long item = next_live(blockIdx.x);
    TcItem cur = {};
    if (item < n_work) cur = tc_decode(P, live_mode, item, s_pref, s_tmax, s_slot0);
    // Cache rows below a row group's smallest position are the requests'
    // committed context, never an output of the previous kernel (that one
    // writes the window's own rows): the first item's 128-key boxes that lie
    // wholly below it are requested before the wait.
    if (threadIdx.x == 0 && item < n_work && live_mode) {
        const int group = cur.tile / P.tiles_per_group;
        const int gmin = s_gmin[group];
        const int nkh = n_keys_of(cur) > 128 ? 2 : 1;
        if (cur.split * SPLIT + nkh * 128 <= gmin) {
            load_kv(&tmK, &tmK2, sK, kbar, k_iss, cur);
            load_kv(&tmV, &tmV2, sV, vbar, v_iss, cur);
            early = 1;
        }
    }
    pdl_wait();
    pdl_trigger();
    if (item < n_work) {
        if (threadIdx.x == 0 && !early) {
            load_kv(&tmK, &tmK2, sK, kbar, k_iss, cur);
            load_kv(&tmV, &tmV2, sV, vbar, v_iss, cur);
        }
        load_q(cur);
    }
    bool ok = true;
#pragma unroll 1
    while (item < n_work) {
        const int key0 = cur.split * SPLIT;
        const int n_keys = n_keys_of(cur);
        const int nkh = n_keys > 128 ? 2 : 1;
        const uint32_t DS = static_cast<uint32_t>(nkh) * 16384u;   // dim-half stride of this item's K / V box
        const int n16 = (n_keys + 15) >> 4;
        int row0, nr;
        tile_rows_of(P, cur.tile, row0, nr);
        const int T = nr * P.G;
        if (threadIdx.x < nr) {
            const int w = row0 + threadIdx.x;
            s_pos[threadIdx.x] = rows_tab ? s_rpos[w] : (row_ok(P, w, cur.slot0) ? P.row_pos[w] : -1);
        }
        const long long nxt_item = next_live(item + gridDim.x);
        const bool has_nxt = nxt_item < n_work;
        TcItem nxt = {};
        if (has_nxt) nxt = tc_decode(P, live_mode, nxt_item, s_pref, s_tmax, s_slot0);

        // ---- Q landed (cp.async, every thread) and visible to the tensor core
        cp_async_wait<0>();
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(aborted())) {
            ok = false;
            break;
        }
        tc_fence_after();
        // ---- S = Q K^T, issued by warp 0: every lane observes the K halves (a
        // time-out anywhere stops all), one elected lane issues the MMAs.
        if (warp == 0) {
            bool got = take(&kbar[0], k_use[0], k_seen[0]);
            got = __all_sync(0xffffffffu, got);
            if (got) {
                tc_fence_after();
                constexpr uint32_t idS = idesc_bf16_f32(M, 128);
                const uint64_t dq = sw128_kmajor_desc(uQ), dk = sw128_kmajor_desc(uK);
#pragma unroll
                for (int kh = 0; kh < 2; ++kh) {
                    if (kh >= nkh) break;
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k) {
                        // start addresses advance in 16-byte units inside the descriptor; keys
                        // 128 kh .. of the box start 16 KiB into each dim half
                        const uint64_t a = dq + static_cast<uint64_t>(((k >> 2) * (M * 128) + (k & 3) * 32) >> 4);
                        const uint64_t b =
                            dk + static_cast<uint64_t>((kh * 16384 + (k >> 2) * DS + (k & 3) * 32) >> 4);
                        umma_bf16_elect(tS + kh * 128, a, b, idS, k > 0 ? 1u : 0u);
                    }
                }
                umma_commit_elect(&sbar);
            } else if (lane == 0) {
                mbar_arrive(&sbar);                        // nothing issued: release the waiters
            }
            ++s_iss;
        }
        ++k_use[0];
        if (mbar_wait(&sbar, s_use & 1u, &abort_flag, &g_attn_err) && threadIdx.x == 0) ++s_seen;
        ++s_use;
        tc_fence_after();
        // ---- S is in TMEM: this item's K may be overwritten (M = 64)
        if (M == 64 && has_nxt && threadIdx.x == 0 && !aborted()) load_kv(&tmK, &tmK2, sK, kbar, k_iss, nxt);

        // ---- softmax over the split, row by row
        const int q4 = warp & 3, ch = warp >> 2;
        const float sl2 = P.scale_log2;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
        const int r = M == 64 ? 16 * q4 + (lane & 15) : 32 * q4 + lane;
        const int hi = M == 64 ? (lane >> 4) : 0;
        const int pos = r < T ? s_pos[r / P.G] : -1;
        // Keys 128 ch + 32 i .. + 31 form chunk i of the thread's half; chunks at
        // or past the split's last key hold no key of any row and are skipped
        // (P V reads P only up to the next 16-key step).
        // The row maximum is taken over the raw scores and scaled once: scaling
        // by sl2 > 0 rounds monotonically, so this equals the maximum of the
        // scaled scores.
        float mraw = -INFINITY;
        // M = 64: the thread's 64 scores (keys 128 ch + 32 i + 16 hi + t) stay in
        // registers from one round of loads until P is written.
        uint32_t sv[4][16];
        if (M == 64) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (128 * ch + 32 * i < n_keys) tmem_ld16x2(tS + lane_base + 128 * ch + 32 * i, sv[i]);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if (128 * ch + 32 * i >= n_keys) continue;
                reg_fence16(sv[i]);
                mraw = fmaxf(mraw, masked_max<16>(sv[i], pos - (key0 + 128 * ch + 32 * i + 16 * hi)));
            }
            mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 16));
        } else {
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int c = 128 * ch + 32 * i;
                if (c >= n_keys) break;
                uint32_t v[32];
                tmem_ld32_sync(tS + lane_base + c, v);
                mraw = fmaxf(mraw, masked_max<32>(v, pos - (key0 + c)));
            }
        }
        float m = __fmul_rn(mraw, sl2);
        if (hi == 0) s_mx[ch][r] = m;
        if (__syncthreads_or(aborted())) {
            ok = false;
            break;
        }
        m = fmaxf(s_mx[0][r], s_mx[1][r]);
        const float nmu = m == -INFINITY ? 0.0f : -m;     // a row with no key in the split
        // l: every 16-key group summed in key order, pairs of groups added, then
        // ((q0 + q1) + (q2 + q3)) per 128-key half and the halves -- the same
        // order for M = 64 and M = 128, so a row's sum never depends on the tile.
        float l = 0.0f;
        float gq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (M == 64) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = 128 * ch + 32 * i;
                if (c >= n_keys) continue;
                const int kc = c + 16 * hi;                   // first key (within the split) of these 16
                uint32_t pk[8];
                // this 16-key group's sum, in key order
                const float lg = softmax_group(sv[i], sl2, nmu, pos - (key0 + kc), pk);
                // groups 2i (hi = 0) and 2i + 1 (hi = 1) of this half: even + odd, in both threads
                const float lo = __shfl_xor_sync(0xffffffffu, lg, 16);
                gq[i] = hi ? lo + lg : lg + lo;
                uint8_t* prow = sP + (kc >> 6) * (M * 128) + r * 128;
                const int pc = (kc & 63) >> 3;
                *reinterpret_cast<uint4*>(prow + ((pc ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4*>(prow + (((pc + 1) ^ (r & 7)) << 4)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            l = (gq[0] + gq[1]) + (gq[2] + gq[3]);
        } else {
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
                const int c = 128 * ch + 32 * i;
                if (c >= n_keys) break;
                uint32_t v[32];
                tmem_ld32_sync(tS + lane_base + c, v);
                uint32_t pk[16];
                const float lg0 = softmax_group(v, sl2, nmu, pos - (key0 + c), pk);
                const float lg1 = softmax_group(v + 16, sl2, nmu, pos - (key0 + c + 16), pk + 8);
                gq[i] = lg0 + lg1;
                uint8_t* prow = sP + (c >> 6) * (M * 128) + r * 128;
                const int pc = (c & 63) >> 3;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(prow + (((pc + q) ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
            l = (gq[0] + gq[1]) + (gq[2] + gq[3]);
        }
        if (hi == 0) s_sum[ch][r] = l;
        if (hi == 0 && ch == 0) s_rowm[r] = m;
        // ---- V rows from the split's last key up to the next 16-key step: zero
        // (a masked p = 0 must never meet a NaN in P V)
        if (warp == 7 && (n_keys & 15) != 0) {
            if (mbar_wait(&vbar[0], v_use[0] & 1u, &abort_flag, &g_attn_err)) {
                for (int idx = lane; idx < (16 * n16 - n_keys) * 16; idx += 32) {
                    const int key = n_keys + (idx >> 4), dh = (idx >> 3) & 1, pc = idx & 7;
                    *reinterpret_cast<uint4*>(sV + dh * DS + key * 128 + pc * 16) = make_uint4(0, 0, 0, 0);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(aborted())) {
            ok = false;
            break;
        }
        tc_fence_after();
        // ---- O = P V, issued by warp 0 like S
        if (warp == 0) {
            bool got = take(&vbar[0], v_use[0], v_seen[0]);
            got = __all_sync(0xffffffffu, got);
            if (got) {
                tc_fence_after();
                constexpr uint32_t idO = idesc_bf16_f32(M, 128) | (1u << 16);   // B (V) MN-major
                const uint64_t dp = sw128_kmajor_desc(uP), dv = sw128_mnmajor_desc(uV, DS);
                for (int st = 0; st < n16; ++st) {
                    const uint64_t a = dp + static_cast<uint64_t>(((st >> 2) * (M * 128) + (st & 3) * 32) >> 4);
                    const uint64_t b = dv + static_cast<uint64_t>((st * 2048) >> 4);
                    umma_bf16_elect(tO, a, b, idO, st > 0 ? 1u : 0u);
                }
                umma_commit_elect(&obar);
            } else if (lane == 0) {
                mbar_arrive(&obar);
            }
            ++o_iss;
        }
        ++v_use[0];
        // the next item's Q (this item's has been read since S landed), while P V runs
        if (has_nxt && !aborted()) load_q(nxt);
        if (mbar_wait(&obar, o_use & 1u, &abort_flag, &g_attn_err) && threadIdx.x == 0) ++o_seen;
        ++o_use;
        tc_fence_after();
        // ---- V (and, for M = 128, K's space, which held P) are free: next loads
        if (threadIdx.x == 0 && has_nxt && !aborted()) {
            fence_proxy_async_smem();
            if (M == 128) load_kv(&tmK, &tmK2, sK, kbar, k_iss, nxt);
            load_kv(&tmV, &tmV2, sV, vbar, v_iss, nxt);
        }
        // ---- the split's partial of every tile row that reaches it
        {
            const int i = r / P.G, g = r - i * P.G;
            const long long ph =
                (static_cast<long long>(row0 + i) * P.Hq + cur.kvh * P.G + g) * P.s_max + cur.split;
            float* dst = P.ws_o + ph * HD;
            if (M == 64) {
                uint32_t ov[2][16];
#pragma unroll
                for (int j = 0; j < 2; ++j) tmem_ld16x2(tO + lane_base + 64 * ch + 32 * j, ov[j]);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    reg_fence16(ov[j]);
                    const uint32_t* v = ov[j];
                    if (pos >= key0) {
                        st_global_v8(dst + 64 * ch + 32 * j + 16 * hi, v);
                        st_global_v8(dst + 64 * ch + 32 * j + 16 * hi + 8, v + 8);
                    }
                }
            } else {
#pragma unroll 1
                for (int j = 0; j < 2; ++j) {
                    const int c = 64 * ch + 32 * j;
                    uint32_t v[32];
                    tmem_ld32_sync(tO + lane_base + c, v);
                    if (pos >= key0) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) st_global_v8(dst + c + 8 * q, v + 8 * q);
                    }
                }
            }
            if (pos >= key0 && ch == 0 && hi == 0) {
                P.ws_m[ph] = s_rowm[r];
                P.ws_l[ph] = s_sum[0][r] + s_sum[1][r];
            }
        }
        tc_fence_before();
        if (__syncthreads_or(aborted())) {              // TMEM, s_mx, s_sum, s_rowm, s_pos are reused
            ok = false;
            break;
        }
        tc_fence_after();
        item = nxt_item;
        cur = nxt;
    }
    // ---- leave.  After a time-out, the copies and MMAs already started
    // complete first (bounded waits), then TMEM is freed.
    cp_async_wait<0>();
    if (threadIdx.x == 0 && !ok) {
        for (int kh = 0; kh < 2; ++kh) {
            for (uint32_t j = k_seen[kh]; j < k_iss[kh]; ++j) mbar_wait_drain(&kbar[kh], j & 1u);
            for (uint32_t j = v_seen[kh]; j < v_iss[kh]; ++j) mbar_wait_drain(&vbar[kh], j & 1u);
        }
        for (uint32_t j = s_seen; j < s_iss; ++j) mbar_wait_drain(&sbar, j & 1u);
        for (uint32_t j = o_seen; j < o_iss; ++j) mbar_wait_drain(&obar, j & 1u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(s_tmem, kTmemCols);
}

// ------------------------------------- two items in flight per SM (M = 64)
// The same work items and the same per-row arithmetic as attn_tc_kernel<64>
// (bit for bit: the same MMAs, maxima, exponentials and summation tree, and
// the same split of every row's keys over two threads of two warps), but
// each CTA runs two warpgroups of eight warps that work through alternate
// items of the CTA's list independently, each with its own shared-memory
// regions, barriers and half of the tensor memory.  Within a warpgroup an
// item is still serial (S -> softmax -> P V -> partials); the other
// warpgroup's item fills the gaps, so two items' loads and latencies overlap
// on every SM.  Per warpgroup (96 KiB):
//   region A (64 KiB): the split's K box for S; then its V box
//   region B (32 KiB): Q (16 KiB) for S; then P (32 KiB)
// and tensor memory columns [256 wg, 256 wg + 256): S, then O in the first
// 128 of them once every thread has read its scores.  The V box is requested
// as soon as S is in TMEM, the next item's K and Q once P V is.
// The tile tables live in dynamic shared memory sized to the call.
constexpr int kPPRegionA = 2 * kTcKeyHalfBytes;       // 64 KiB: K, then V
constexpr int kPPRegionB = kTcKeyHalfBytes;           // 32 KiB: Q, then P
constexpr int kPPGroup = kPPRegionA + kPPRegionB;     // per warpgroup
constexpr int kPPWGThreads = 256;                     // per warpgroup
constexpr int kPPThreads = 2 * kPPWGThreads;

// Ints of the tile tables for n_tiles tiles and W rows: largest position,
// prefix sums (+ total), first slot and smallest group position per tile,
// each row's position, the warp sums of the scan.
inline long long pp_table_ints(long long n_tiles, long long W) { return 4 * n_tiles + 1 + W + ATTN_THREADS / 32; }
inline size_t pp_smem_bytes(long long n_tiles, long long W) {
    return 1024 + 2 * static_cast<size_t>(kPPGroup) + static_cast<size_t>(pp_table_ints(n_tiles, W)) * 4;
}
constexpr size_t kPPSmemMax = 224 * 1024;                 // + the kernel's static shared memory <= 227 KiB

// Barrier over the 256 threads of warpgroup wg that ORs a flag across them.
BIV_DEV bool wg_sync_or(int wg, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(1 + wg)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kPPThreads, 1)
attn_pp_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ CUtensorMap tmK2, const __grid_constant__ CUtensorMap tmV2,
               const __grid_constant__ CUtensorMap tmQ, const AttnParams P) {
    constexpr int M = 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp >> 3;                         // warpgroup
    const int w8 = warp & 7;                          // warp within the warpgroup
    const int wt = threadIdx.x & (kPPWGThreads - 1);  // thread within the warpgroup
    const int q4 = w8 & 3, ch = w8 >> 2;              // TMEM lane quarter, 128-key half of the split
    uint8_t* sA = smem + wg * kPPGroup;               // K, then V
    uint8_t* sB = sA + kPPRegionA;                    // Q, then P
    const uint32_t uA = smem_u32(sA), uB = smem_u32(sB);
    const int n_tiles = P.n_tiles;
    int* s_tmax = reinterpret_cast<int*>(smem + 2 * kPPGroup);
    int* s_pref = s_tmax + n_tiles;                   // n_tiles + 1
    int* s_slot0 = s_pref + n_tiles + 1;
    int* s_gmin = s_slot0 + n_tiles;
    int* s_rpos = s_gmin + n_tiles;
    int* s_wsum = s_rpos + P.W;

    __shared__ __align__(8) uint64_t kbar[2][2], vbar[2][2], qbar[2], sbar[2], obar[2];
    __shared__ uint32_t s_tmem;
    __shared__ int abort_flag;
    __shared__ uint32_t s_qiss[2], s_viss[2];
    __shared__ float s_mx[2][2][M], s_sum[2][2][M];

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int g = 0; g < 2; ++g) {
            for (int i = 0; i < 2; ++i) {
                mbar_init(&kbar[g][i], 1);
                mbar_init(&vbar[g][i], 1);
            }
            mbar_init(&qbar[g], 1);
            mbar_init(&sbar[g], 1);
            mbar_init(&obar[g], 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, kTmemCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmK2);
        prefetch_tensormap(&tmV2);
        prefetch_tensormap(&tmQ);
    }
    tc_fence_before();
    // The tables read only the window's slots and positions (inputs of the
    // call): built while the previous kernel finishes.
    build_tile_tables(P, s_tmax, s_pref, s_slot0, s_wsum, s_rpos, s_gmin, n_tiles, P.W);   // ends with a barrier
    tc_fence_after();
    const uint32_t tS = s_tmem + 256u * static_cast<uint32_t>(wg), tO = tS;
    const long long n_work = s_pref[n_tiles];
    const long long step = 2LL * gridDim.x;

    uint64_t* kb = kbar[wg];
    uint64_t* vb = vbar[wg];
    uint32_t k_use[2] = {0u, 0u}, v_use[2] = {0u, 0u}, s_use = 0u, o_use = 0u, q_use = 0u;
    uint32_t k_iss[2] = {0u, 0u}, v_iss[2] = {0u, 0u}, s_iss = 0u, o_iss = 0u, q_iss = 0u;
    uint32_t k_seen[2] = {0u, 0u}, v_seen[2] = {0u, 0u}, s_seen = 0u, o_seen = 0u, q_seen = 0u;
    uint32_t early = 0;

    auto n_keys_of = [&](const TcItem& it) { return min(SPLIT, it.maxpos + 1 - it.split * SPLIT); };
    auto kv_row_of = [&](const TcItem& it) { return (it.slot0 * P.Hkv + it.kvh) * P.max_len + it.split * SPLIT; };
    // warpgroup thread 0: the K or V of an item as one box ([2 dim halves][R
    // keys][128 B], R = 256 for a split with more than 128 keys, else 128)
    auto load_box = [&](const CUtensorMap* map, const CUtensorMap* map2, uint8_t* dst, uint64_t* bar, uint32_t& iss,
                        const TcItem& it) {
        const int nkh = n_keys_of(it) > 128 ? 2 : 1;
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nkh * kTcKeyHalfBytes));
        tma_load_3d(dst, nkh == 2 ? map2 : map, bar, 0, kv_row_of(it), 0, policy_evict_first());
        ++iss;
    };
    // warpgroup thread 0: the item's Q tile into region B as two 4-D boxes,
    // one per 64-dim half ([tile rows][G heads][128 B]: tile row i * G + g,
    // K-major, 128-byte swizzle, the halves M * 128 B apart as the S MMA reads
    // them); rows past the window are zero-filled, rows of the next group are
    // loaded but never used.
    const uint32_t q_bytes = static_cast<uint32_t>(P.tile_rows * P.G * HD * 2);
    auto load_q = [&](const TcItem& it) {
        int row0, nr;
        tile_rows_of(P, it.tile, row0, nr);
        mbar_arrive_expect_tx(&qbar[wg], q_bytes);
        tma_load_4d(sB, &tmQ, &qbar[wg], 0, it.kvh * P.G, row0, 0, policy_evict_first());
        tma_load_4d(sB + M * 128, &tmQ, &qbar[wg], 0, it.kvh * P.G, row0, 1, policy_evict_first());
        ++q_iss;
    };
    auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&abort_flag) != 0; };
    auto take = [&](uint64_t* bar, uint32_t use, uint32_t& seen) {
        const bool got = mbar_wait(bar, use & 1u, &abort_flag, &g_attn_err, true);
        if (got) ++seen;
        return got;
    };

    long long item = static_cast<long long>(blockIdx.x) + static_cast<long long>(wg) * gridDim.x;
    TcItem cur = {};
    if (item < n_work) cur = tc_decode(P, true, item, s_pref, s_tmax, s_slot0);
    // K boxes of the first item that lie wholly below its row group's smallest
    // position (committed context, not the previous kernel's output): before the wait
    if (wt == 0 && item < n_work) {
        const int gmin = s_gmin[cur.tile / P.tiles_per_group];
        const int nkh = n_keys_of(cur) > 128 ? 2 : 1;
        if (cur.split * SPLIT + nkh * 128 <= gmin) {
            load_box(&tmK, &tmK2, sA, &kb[0], k_iss[0], cur);
            early = 1;
        }
    }
    pdl_wait();
    pdl_trigger();
    if (item < n_work && wt == 0 && !early) load_box(&tmK, &tmK2, sA, &kb[0], k_iss[0], cur);
    if (item < n_work && wt == 32) load_q(cur);
    const float sl2 = P.scale_log2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const int r = 16 * q4 + (lane & 15);              // the thread's tile row
    const int hi = lane >> 4;
    bool ok = true;
#pragma unroll 1
    while (item < n_work) {
        const int key0 = cur.split * SPLIT;
        const int n_keys = n_keys_of(cur);
        const int nkh = n_keys > 128 ? 2 : 1;
        const uint32_t DS = static_cast<uint32_t>(nkh) * 16384u;   // dim-half stride of this item's K / V box
        const int n16 = (n_keys + 15) >> 4;
        int row0, nr;
        tile_rows_of(P, cur.tile, row0, nr);
        const int T = nr * P.G;
        const long long nxt_item = item + step;
        const bool has_nxt = nxt_item < n_work;
        TcItem nxt = {};
        if (has_nxt) nxt = tc_decode(P, true, nxt_item, s_pref, s_tmax, s_slot0);

        // ---- S = Q K^T by the warpgroup's first warp (one elected lane), once
        // the item's Q and K boxes have landed
        if (w8 == 0) {
            bool got = take(&qbar[wg], q_use, q_seen) && take(&kb[0], k_use[0], k_seen[0]);
            got = __all_sync(0xffffffffu, got);
            if (got) {
                tc_fence_after();
                constexpr uint32_t idS = idesc_bf16_f32(M, 128);
                const uint64_t dq = sw128_kmajor_desc(uB), dk = sw128_kmajor_desc(uA);
#pragma unroll
                for (int kh = 0; kh < 2; ++kh) {
                    if (kh >= nkh) break;
#pragma unroll
                    for (int k = 0; k < HD / 16; ++k) {
                        const uint64_t a = dq + static_cast<uint64_t>(((k >> 2) * (M * 128) + (k & 3) * 32) >> 4);
                        const uint64_t b = dk + static_cast<uint64_t>((kh * 16384 + (k >> 2) * DS + (k & 3) * 32) >> 4);
                        umma_bf16_elect(tS + kh * 128, a, b, idS, k > 0 ? 1u : 0u);
                    }
                }
                umma_commit_elect(&sbar[wg]);
            } else if (lane == 0) {
                mbar_arrive(&sbar[wg]);                    // nothing issued: release the waiters
            }
            ++s_iss;
        }
        ++k_use[0];
        ++q_use;
        if (mbar_wait(&sbar[wg], s_use & 1u, &abort_flag, &g_attn_err) && wt == 0) ++s_seen;
        ++s_use;
        tc_fence_after();
        // ---- Q and K consumed: this item's V box into region A, issued by
        // warp 7 (warp 0 has just issued the S MMAs and will issue P V)
        if (wt == 224 && !aborted()) load_box(&tmV, &tmV2, sA, &vb[0], v_iss[0], cur);
        // ---- softmax over the split; the thread's 64 scores (keys 128 ch + 32 i
        // + 16 hi + t) stay in registers from one round of loads until P is written
        const int pos = r < T ? s_rpos[row0 + r / P.G] : -1;     // the row's usable position (table)
        float mraw = -INFINITY;
        uint32_t sv[4][16];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (128 * ch + 32 * i < n_keys) tmem_ld16x2(tS + lane_base + 128 * ch + 32 * i, sv[i]);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (128 * ch + 32 * i >= n_keys) continue;
            reg_fence16(sv[i]);
            mraw = fmaxf(mraw, masked_max<16>(sv[i], pos - (key0 + 128 * ch + 32 * i + 16 * hi)));
        }
        mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 16));
        float m = __fmul_rn(mraw, sl2);
        if (hi == 0) s_mx[wg][ch][r] = m;
        if (wg_sync_or(wg, aborted())) {
            ok = false;
            break;
        }
        m = fmaxf(s_mx[wg][0][r], s_mx[wg][1][r]);
        const float nmu = m == -INFINITY ? 0.0f : -m;      // a row with no key in the split
        // l: every 16-key group summed in key order, pairs of groups added, then
        // ((q0 + q1) + (q2 + q3)) per 128-key half and the halves
        float gq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = 128 * ch + 32 * i;
            if (c >= n_keys) continue;
            const int kc = c + 16 * hi;
            uint32_t pk[8];
            const float lg = softmax_group(sv[i], sl2, nmu, pos - (key0 + kc), pk);
            const float lo = __shfl_xor_sync(0xffffffffu, lg, 16);
            gq[i] = hi ? lo + lg : lg + lo;
            uint8_t* prow = sB + (kc >> 6) * (M * 128) + r * 128;
            const int pc = (kc & 63) >> 3;
            *reinterpret_cast<uint4*>(prow + ((pc ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(prow + (((pc + 1) ^ (r & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        if (hi == 0) s_sum[wg][ch][r] = (gq[0] + gq[1]) + (gq[2] + gq[3]);
        // ---- V rows from the split's last key up to the next 16-key step: zero
        if (w8 == 7 && (n_keys & 15) != 0) {
            if (mbar_wait(&vb[0], v_use[0] & 1u, &abort_flag, &g_attn_err)) {
                for (int idx = lane; idx < (16 * n16 - n_keys) * 16; idx += 32) {
                    const int key = n_keys + (idx >> 4), dh = (idx >> 3) & 1, pc = idx & 7;
                    *reinterpret_cast<uint4*>(sA + dh * DS + key * 128 + pc * 16) = make_uint4(0, 0, 0, 0);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (wg_sync_or(wg, aborted())) {               // P written; every thread has read its S
            ok = false;
            break;
        }
        tc_fence_after();
        // ---- O = P V into the first 128 columns of the S region
        if (w8 == 0) {
            bool got = take(&vb[0], v_use[0], v_seen[0]);
            got = __all_sync(0xffffffffu, got);
            if (got) {
                tc_fence_after();
                constexpr uint32_t idO = idesc_bf16_f32(M, 128) | (1u << 16);   // B (V) MN-major
                const uint64_t dp = sw128_kmajor_desc(uB), dv = sw128_mnmajor_desc(uA, DS);
                for (int st = 0; st < n16; ++st) {
                    const uint64_t a = dp + static_cast<uint64_t>(((st >> 2) * (M * 128) + (st & 3) * 32) >> 4);
                    const uint64_t b = dv + static_cast<uint64_t>((st * 2048) >> 4);
                    umma_bf16_elect(tO, a, b, idO, st > 0 ? 1u : 0u);
                }
                umma_commit_elect(&obar[wg]);
            } else if (lane == 0) {
                mbar_arrive(&obar[wg]);
            }
            ++o_iss;
        }
        ++v_use[0];
        if (mbar_wait(&obar[wg], o_use & 1u, &abort_flag, &g_attn_err) && wt == 0) ++o_seen;
        ++o_use;
        tc_fence_after();
        // ---- P and V consumed: the next item's K and Q, issued by two
        // threads of two warps (an issue waits while the copy engine is busy)
        if (has_nxt && !aborted() && (wt == 0 || wt == 32)) {
            fence_proxy_async_smem();
            if (wt == 0)
                load_box(&tmK, &tmK2, sA, &kb[0], k_iss[0], nxt);
            else
                load_q(nxt);
        }
        // ---- the split's partial of every tile row that reaches it
        {
            const int i = r / P.G, g = r - i * P.G;
            const long long ph = (static_cast<long long>(row0 + i) * P.Hq + cur.kvh * P.G + g) * P.s_max + cur.split;
            float* dst = P.ws_o + ph * HD;
            uint32_t ov[2][16];
#pragma unroll
            for (int j = 0; j < 2; ++j) tmem_ld16x2(tO + lane_base + 64 * ch + 32 * j, ov[j]);
            tmem_ld_wait();
            // O is in registers: the TMEM columns may take the next item's S
            // while these stores drain
            tc_fence_before();
            if (wg_sync_or(wg, aborted())) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                reg_fence16(ov[j]);
                const uint32_t* v = ov[j];
                if (pos >= key0) {
                    st_global_v8(dst + 64 * ch + 32 * j + 16 * hi, v);
                    st_global_v8(dst + 64 * ch + 32 * j + 16 * hi + 8, v + 8);
                }
            }
            if (pos >= key0 && ch == 0 && hi == 0) {
                P.ws_m[ph] = m;
                P.ws_l[ph] = s_sum[wg][0][r] + s_sum[wg][1][r];
            }
        }
        item = nxt_item;
        cur = nxt;
    }
    // ---- leave.  After a time-out, the copies and MMAs already started
    // complete first (bounded waits), then TMEM is freed.  (ok is uniform
    // over the warpgroup; threads 32 and 224 issued the Q and V boxes, thread 0
    // saw them land.)
    if (!ok) {
        if (wt == 32) s_qiss[wg] = q_iss;
        if (wt == 224) s_viss[wg] = v_iss[0];
        asm volatile("bar.sync %0, 256;" ::"r"(1 + wg) : "memory");
    }
    if (wt == 0 && !ok) {
        for (uint32_t j = q_seen; j < s_qiss[wg]; ++j) mbar_wait_drain(&qbar[wg], j & 1u);
        for (uint32_t j = k_seen[0]; j < k_iss[0]; ++j) mbar_wait_drain(&kb[0], j & 1u);
        for (uint32_t j = v_seen[0]; j < s_viss[wg]; ++j) mbar_wait_drain(&vb[0], j & 1u);
        for (uint32_t j = s_seen; j < s_iss; ++j) mbar_wait_drain(&sbar[wg], j & 1u);
        for (uint32_t j = o_seen; j < o_iss; ++j) mbar_wait_drain(&obar[wg], j & 1u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(s_tmem, kTmemCols);
}

// One warp per (row, head): combine splits 0 .. pos/256 of the row.  Lane s
// holds split s (32 at a time); the maximum and the weight sum are reduced
// with a fixed xor butterfly, the outputs are summed in increasing split
// order.  Per pair one round of loads fetches the (m, l) of up to 64 splits
// and the first kCombinePre splits' outputs together; the later splits come
// kCombinePre at a time (a pair of 33 splits: five rounds of loads).
//
// Which warp combines which pair does not change a pair's arithmetic, so the
// pairs are dealt for balance.  A pair of ns splits costs kCombinePre units
// per round of loads plus one per split: the bulk of the combine runs near
// the HBM rate, where bytes count, and its tail is a few warps' chains of
// rounds, where rounds count.  A pair that is only zeroed costs one unit.
// Every CTA forms the prefix sums of the rows' costs from the call's slots
// and positions (inputs, so before the wait on the split kernel), and warp g
// of NW takes the pairs whose cost interval starts in [T·g/NW, T·(g+1)/NW).
// With lognormal context lengths a fixed round-robin deal gave some warps
// twice the mean work.  Windows of more than kCombineBalancedMaxW rows (whose
// cost table would not fit beside three CTAs per SM) keep the round-robin
// deal.
constexpr int kCombinePre = 8;
constexpr int kCombineBalancedMaxW = 4096;

// A pair's cost in the balanced deal (ns = 0: a pair that is only zeroed).
__host__ __device__ inline int combine_cost(int ns) {
    return ns > 0 ? kCombinePre * ((ns + kCombinePre - 1) / kCombinePre) + ns : 1;
}

// The balanced deal is used where warps have several pairs each (with about
// one pair per warp, round-robin gives every warp a single pair and the
// balanced deal could give a warp two), its tables fit in shared memory and
// its 32-bit cost sums cannot overflow (a pair costs at most 2·s_max + kCombinePre).
constexpr int kCombineBalancedMinPairsPerWarp = 4;
__host__ __device__ inline bool combine_balanced(int W, int Hq, int s_max, int n_warps) {
    return W <= kCombineBalancedMaxW &&
           static_cast<long long>(W) * Hq >= static_cast<long long>(kCombineBalancedMinPairsPerWarp) * n_warps &&
           static_cast<long long>(W) * Hq * (2ll * s_max + kCombinePre) < (1ll << 31);
}

// Shared-memory bytes of the balanced deal's tables (0: round-robin deal).
inline size_t combine_smem_bytes(int W, int Hq, int s_max, int n_warps) {
    return combine_balanced(W, Hq, s_max, n_warps) ? static_cast<size_t>(2 * W + 1) * sizeof(int) : 0;
}

struct CombineRow {
    int slot, pos, slot0;
};

BIV_DEV CombineRow combine_row(const AttnParams& P, long long pair) {
    const int w = static_cast<int>(pair / P.Hq);
    const int grp0 = (w / P.rows_per_group) * P.rows_per_group;
    return CombineRow{P.row_slot[w], P.row_pos[w], P.row_slot[grp0]};
}

// Splits to combine for a row (0: the row is not attended and its output is zero).
BIV_DEV int combine_splits(const AttnParams& P, const CombineRow& rw) {
    const int p = rw.pos;
    if (rw.slot < 0 || rw.slot >= P.n_slots || p < 0 || p >= P.max_len || rw.slot != rw.slot0) return 0;
    return p / SPLIT + 1;
}

// The whole warp combines pair `pair` over its ns splits (ns = 0: zeros).
BIV_DEV void combine_pair(const AttnParams& P, __nv_bfloat16* __restrict__ out, long long pair, int ns, int lane) {
    __nv_bfloat16* dst = out + pair * HD + lane * 4;
    if (ns <= 0) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
        return;
    }
    const long long base = pair * P.s_max;
    const float4* src0 = reinterpret_cast<const float4*>(P.ws_o + base * HD) + lane;
    float4 pre[kCombinePre];
#pragma unroll
    for (int j = 0; j < kCombinePre; ++j)
        pre[j] = j < ns ? src0[static_cast<long long>(j) * (HD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
    // (m, l) of the first 64 splits in the same round (a pair of 33 splits,
    // from a context of 8192, would otherwise wait twice more for split 33's)
    const float m0 = lane < ns ? P.ws_m[base + lane] : -INFINITY;
    const float l0 = lane < ns ? P.ws_l[base + lane] : 0.0f;
    const float m1 = 32 + lane < ns ? P.ws_m[base + 32 + lane] : -INFINITY;
    const float l1 = 32 + lane < ns ? P.ws_l[base + 32 + lane] : 0.0f;
    // Row maximum over all splits.
    float M = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 32) {
        float m = s0 == 0 ? m0 : s0 == 32 ? m1 : (s0 + lane < ns) ? P.ws_m[base + s0 + lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        M = fmaxf(M, m);
    }
    float L = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 32) {
        const int s = s0 + lane;
        const float ms = s0 == 0 ? m0 : s0 == 32 ? m1 : (s < ns) ? P.ws_m[base + s] : -INFINITY;
        const float ls = s0 == 0 ? l0 : s0 == 32 ? l1 : (s < ns) ? P.ws_l[base + s] : 0.0f;
        const float wgt = (s < ns) ? exp2f(ms - M) : 0.0f;
        float lw = (s < ns) ? wgt * ls : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        L += lw;
        const int cnt = min(32, ns - s0);
        const float4* src = src0 + static_cast<long long>(s0) * (HD / 4);
        for (int j0 = 0; j0 < cnt; j0 += kCombinePre) {
            if (s0 > 0 || j0 > 0) {
                // the next kCombinePre splits in one round of loads (the first
                // ones were prefetched above)
#pragma unroll
                for (int q = 0; q < kCombinePre; ++q)
                    pre[q] = j0 + q < cnt ? src[static_cast<long long>(j0 + q) * (HD / 4)]
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // summed in increasing split order, indexed statically (warp-uniform guard)
#pragma unroll
            for (int q = 0; q < kCombinePre; ++q) {
                if (j0 + q < cnt) {
                    const float wj = __shfl_sync(0xffffffffu, wgt, j0 + q);
                    acc.x += wj * pre[q].x;
                    acc.y += wj * pre[q].y;
                    acc.z += wj * pre[q].z;
                    acc.w += wj * pre[q].w;
                }
            }
        }
    }
    const float inv = 1.0f / L;
    uint2 r;
    r.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    r.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = r;
}

__global__ void __launch_bounds__(256)
attn_combine_kernel(const AttnParams P, __nv_bfloat16* __restrict__ out) {
    extern __shared__ int s_comb[];             // balanced deal: [W + 1] prefix costs, [W] splits per row
    const int W = P.W, Hq = P.Hq;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_warps = static_cast<int>(gridDim.x) * 8;
    const int gw = static_cast<int>(blockIdx.x) * 8 + warp;
    if (combine_balanced(W, Hq, P.s_max, n_warps)) {
        int* s_cum = s_comb;
        int* s_ns = s_comb + W + 1;
        __shared__ int s_wsum[8];
        // each thread a contiguous run of rows: their splits and cost
        const int per = (W + 255) / 256;
        const int r0 = min(W, static_cast<int>(threadIdx.x) * per), r1 = min(W, r0 + per);
        int sum = 0;
        for (int i = r0; i < r1; ++i) {
            const int w = i;
            const int grp0 = (w / P.rows_per_group) * P.rows_per_group;
            const int ns = combine_splits(P, CombineRow{P.row_slot[w], P.row_pos[w], P.row_slot[grp0]});
            s_ns[i] = ns;
            sum += Hq * combine_cost(ns);
        }
        // exclusive prefix of the threads' sums: warp scan, then the warps' totals
        int inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) s_wsum[warp] = inc;
        __syncthreads();
        int run = inc - sum;
        for (int k = 0; k < warp; ++k) run += s_wsum[k];
        for (int i = r0; i < r1; ++i) {
            s_cum[i] = run;
            run += Hq * combine_cost(s_ns[i]);
        }
        if (threadIdx.x == 255) s_cum[W] = run;     // the last thread's run ends at the total
        __syncthreads();
        pdl_wait();
        pdl_trigger();
        const long long T = s_cum[W];
        const long long lo = T * gw / n_warps, hi = T * (gw + 1) / n_warps;
        // the last row whose cost interval starts at or before lo
        int a = 0, b = W - 1;
        while (a < b) {
            const int m = (a + b + 1) >> 1;
            if (s_cum[m] <= lo) a = m;
            else b = m - 1;
        }
        int i = a;
        int u = combine_cost(s_ns[i]);
        int h = static_cast<int>((lo - s_cum[i] + u - 1) / u);   // first head starting at or after lo
        if (h >= Hq) {
            ++i;
            h = 0;
        }
#pragma unroll 1
        while (i < W) {
            u = combine_cost(s_ns[i]);
            if (s_cum[i] + static_cast<long long>(h) * u >= hi) break;
            combine_pair(P, out, static_cast<long long>(i) * Hq + h, s_ns[i], lane);
            if (++h == Hq) {
                h = 0;
                ++i;
            }
        }
        return;
    }
    // round-robin deal: warp g takes pairs g, g + NW, ...; lane i holds the
    // row of the warp's pair first + i * NW (32 at a time)
    const long long n_pairs = static_cast<long long>(W) * Hq;
    const long long first = gw;
    const long long stride = n_warps;
    CombineRow mine = first + lane * stride < n_pairs ? combine_row(P, first + lane * stride)
                                                      : CombineRow{-1, -1, -1};
    pdl_wait();
    pdl_trigger();
    int k = 0;
#pragma unroll 1
    for (long long pair = first; pair < n_pairs; pair += stride, ++k) {
        if (k == 32) {
            k = 0;
            const long long pl = pair + lane * stride;
            mine = pl < n_pairs ? combine_row(P, pl) : CombineRow{-1, -1, -1};
        }
        const CombineRow rw{__shfl_sync(0xffffffffu, mine.slot, k), __shfl_sync(0xffffffffu, mine.pos, k),
                            __shfl_sync(0xffffffffu, mine.slot0, k)};
        combine_pair(P, out, pair, combine_splits(P, rw), lane);
    }
}

// ------------------------------------------------------------------ RoPE
__global__ void rope_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ q_out,
                            __nv_bfloat16* __restrict__ k_out, const int32_t* __restrict__ row_pos, int W,
                            int Hq, int Hkv, int hd, float theta) {
    pdl_wait();
    pdl_trigger();
    const int half = hd / 2;
    const long long total = static_cast<long long>(W) * (Hq + Hkv) * half;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(idx % half);
        const long long rh = idx / half;
        const int h = static_cast<int>(rh % (Hq + Hkv));
        const int w = static_cast<int>(rh / (Hq + Hkv));
        const __nv_bfloat16* src = qkv + (static_cast<long long>(w) * (Hq + 2 * Hkv) + h) * hd;
        __nv_bfloat16* dst = h < Hq ? q_out + (static_cast<long long>(w) * Hq + h) * hd
                                    : k_out + (static_cast<long long>(w) * Hkv + (h - Hq)) * hd;
        rope_rotate(__bfloat162float(src[i]), __bfloat162float(src[i + half]), row_pos[w], i, hd, theta, dst + i,
                    dst + i + half);
    }
}

// RoPE on q and k of one row, with the rotated k and the v of the row written
// straight into the caches at (row_slot, row_pos) -- the verifier's KV
// overwrite in the same pass.  One CTA per row.
__global__ void rope_kv_write_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ q_out,
                                     __nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc,
                                     const int32_t* __restrict__ row_slot, const int32_t* __restrict__ row_pos,
                                     const int32_t* __restrict__ rows_keep, int K, int Hq, int Hkv, int hd,
                                     int n_slots, int max_len, float theta) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x;
    const int half = hd / 2;
    const int pos = row_pos[w], slot = row_slot[w];
    const __nv_bfloat16* src = qkv + static_cast<long long>(w) * (Hq + 2 * Hkv) * hd;
    const bool keep = !rows_keep || (w % K) < rows_keep[w / K];
    const bool cache_ok = slot >= 0 && slot < n_slots && pos >= 0 && pos < max_len;
    if (keep && !cache_ok && threadIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
    const bool write_kv = keep && cache_ok;
    for (int idx = threadIdx.x; idx < (Hq + Hkv) * half; idx += blockDim.x) {
        const int h = idx / half, i = idx - h * half;
        const __nv_bfloat16* x = src + static_cast<long long>(h) * hd;
        __nv_bfloat16* dst;
        if (h < Hq) {
            dst = q_out + (static_cast<long long>(w) * Hq + h) * hd;
        } else {
            if (!write_kv) continue;
            dst = kc + ((static_cast<long long>(slot) * Hkv + (h - Hq)) * max_len + pos) * hd;
        }
        rope_rotate(__bfloat162float(x[i]), __bfloat162float(x[i + half]), pos, i, hd, theta, dst + i, dst + i + half);
    }
    if (write_kv) {
        const int chunks = Hkv * hd / 8;
        for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
            const int h = c / (hd / 8), e = (c % (hd / 8)) * 8;
            *reinterpret_cast<uint4*>(vc + ((static_cast<long long>(slot) * Hkv + h) * max_len + pos) * hd + e) =
                *reinterpret_cast<const uint4*>(src + static_cast<long long>(Hq + Hkv + h) * hd + e);
        }
    }
}

// ---------------------------------------------------------- KV overwrite
__global__ void kv_overwrite_kernel(__nv_bfloat16* __restrict__ kc, __nv_bfloat16* __restrict__ vc,
                                    const __nv_bfloat16* __restrict__ k_new, long long k_stride,
                                    const __nv_bfloat16* __restrict__ v_new, long long v_stride,
                                    const int32_t* __restrict__ row_slot,
                                    const int32_t* __restrict__ row_pos, const int32_t* __restrict__ rows_keep,
                                    int K, int Hkv, int hd, int n_slots, int max_len) {
    pdl_wait();
    pdl_trigger();
    const int w = blockIdx.x;
    const int slot = row_slot[w], p = row_pos[w];
    if (rows_keep && (w % K) >= rows_keep[w / K]) return;
    if (slot < 0 || slot >= n_slots || p < 0 || p >= max_len) {
        if (threadIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
        return;
    }
    const int chunks = Hkv * hd / 8;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const int h = c / (hd / 8), e = (c % (hd / 8)) * 8;
        const long long dst = ((static_cast<long long>(slot) * Hkv + h) * max_len + p) * hd + e;
        const long long off = static_cast<long long>(h) * hd + e;
        *reinterpret_cast<uint4*>(kc + dst) = *reinterpret_cast<const uint4*>(k_new + w * k_stride + off);
        *reinterpret_cast<uint4*>(vc + dst) = *reinterpret_cast<const uint4*>(v_new + w * v_stride + off);
    }
}

long long splits_for(int max_len) { return (static_cast<long long>(max_len) + SPLIT - 1) / SPLIT; }

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" size_t biv_decode_attn_workspace_size(int W, int Hq, int max_len) {
    if (W <= 0 || Hq <= 0 || max_len <= 0) return 0;
    const long long pairs = static_cast<long long>(W) * Hq * splits_for(max_len);
    return static_cast<size_t>(pairs) * (HD + 2) * sizeof(float) + 16;   // + room to align the partials to 32 B
}

extern "C" int biv_gqa_max_drafts(int G, int tile) {
    BIV_TRACE_CALL();
    if (G <= 0 || G > tile) return -1;
    return tile / G - 1;
}

extern "C" int biv_decode_attn_fixedsplit(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* row_slot, const int32_t* row_pos, void* o, int W,
                                          int rows_per_group, int Hq, int Hkv, int hd, int n_slots, int max_len,
                                          int kv_split, void* workspace, size_t ws_bytes, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || Hq <= 0 || Hkv <= 0 || n_slots <= 0 || max_len <= 0 || rows_per_group <= 0)
        return BIV_ERR_SHAPE;
    if (hd != HD || kv_split != SPLIT) return BIV_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0 || Hq / Hkv > BIV_ATTN_TILE) return BIV_ERR_SHAPE;
    if (W == 0) return BIV_OK;
    if (!q || !k_cache || !v_cache || !row_slot || !row_pos || !o || !workspace) return BIV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
        return BIV_ERR_ALIGN;
    if (ws_bytes < biv_decode_attn_workspace_size(W, Hq, max_len)) return BIV_ERR_SHAPE;
    const long long s_max = splits_for(max_len);
    if (s_max > 65535) return BIV_ERR_SHAPE;

    AttnParams P;
    P.q = static_cast<const __nv_bfloat16*>(q);
    P.kc = static_cast<const __nv_bfloat16*>(k_cache);
    P.vc = static_cast<const __nv_bfloat16*>(v_cache);
    P.row_slot = row_slot;
    P.row_pos = row_pos;
    const long long pairs = static_cast<long long>(W) * Hq * s_max;
    // partial outputs 32-byte aligned (whole-sector stores)
    P.ws_o = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(workspace) + 31) & ~static_cast<uintptr_t>(31));
    P.ws_m = P.ws_o + pairs * HD;
    P.ws_l = P.ws_m + pairs;
    P.W = W;
    P.G = Hq / Hkv;
    P.rows_per_group = std::min(rows_per_group, W);
    P.tile_rows = std::min(P.rows_per_group, BIV_ATTN_TILE / P.G);
    P.tiles_per_group = (P.rows_per_group + P.tile_rows - 1) / P.tile_rows;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.n_slots = n_slots;
    P.max_len = max_len;
    P.s_max = static_cast<int>(s_max);
    P.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));

    const long long n_groups = (W + P.rows_per_group - 1) / P.rows_per_group;
    const long long n_tiles = n_groups * P.tiles_per_group;
    if (n_tiles > 0x7fffffffLL / 64 || Hkv > 65535) return BIV_ERR_SHAPE;
    P.n_tiles = static_cast<int>(n_tiles);
    // K and V caches as TMA sees them: [2 halves of a row][n_slots*Hkv*max_len rows][64 elements]
    // K and V caches as TMA sees them: [2 halves of a row][n_slots*Hkv*max_len
    // rows][64 elements]; boxes of 128 keys (tk, tv) and of a whole 256-key
    // split (tk2, tv2), each landing as [2 dim halves][keys][128 B]
    CUtensorMap tk, tv, tk2, tv2;
    {
        EncodeTiledFn enc = encode_fn();
        if (!enc) {
            set_cuda_error(cudaErrorNotSupported);
            return BIV_ERR_CUDA;
        }
        cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(n_slots) * Hkv * max_len, 2};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(ROWB), 128};
        cuuint32_t es[3] = {1, 1, 1};
        const void* bases[4] = {k_cache, v_cache, k_cache, v_cache};
        CUtensorMap* maps[4] = {&tk, &tv, &tk2, &tv2};
        for (int i = 0; i < 4; ++i) {
            cuuint32_t box[3] = {64, i < 2 ? 128u : 256u, 2};
            if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(bases[i]), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                set_cuda_error(cudaErrorInvalidValue);
                return BIV_ERR_CUDA;
            }
        }
    }

    // Q as TMA sees it for the two-item kernel: [2 dim halves][W rows][Hq
    // heads][64 elements]; a box is one dim half of a tile: [tile rows][G
    // heads][64], i.e. tile row i * G + g
    CUtensorMap tq;
    {
        EncodeTiledFn enc = encode_fn();
        cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(W), 2};
        cuuint64_t strides[3] = {static_cast<cuuint64_t>(ROWB), static_cast<cuuint64_t>(Hq) * ROWB, 128};
        cuuint32_t box[4] = {64, static_cast<cuuint32_t>(P.G), static_cast<cuuint32_t>(P.tile_rows), 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            set_cuda_error(cudaErrorInvalidValue);
            return BIV_ERR_CUDA;
        }
    }
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_status(de);
    int combine_per_sm = 0;                        // resident combine CTAs per SM
    {
        // once per device, from any host thread: kernel attributes and occupancy
        static std::mutex mu;
        static int per_sm[kMaxDevices] = {};       // 0 = not yet configured
        if (dev < 0 || dev >= kMaxDevices) return BIV_ERR_DEVICE;
        std::lock_guard<std::mutex> lock(mu);
        if (per_sm[dev] == 0) {
            cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(tc_smem_bytes<64>()));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(tc_smem_bytes<128>()));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(attn_pp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPPSmemMax));
            if (e != cudaSuccess) return cuda_status(e);
            int per = 0;
            // with the balanced deal's largest tables
            const size_t comb_smem = static_cast<size_t>(2 * kCombineBalancedMaxW + 1) * sizeof(int);
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, attn_combine_kernel, 256, comb_smem) !=
                    cudaSuccess ||
                per < 1)
                per = 1;
            per_sm[dev] = per;
        }
        combine_per_sm = per_sm[dev];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long n_items = static_cast<long long>(s_max) * Hkv * n_tiles;
    const int grid = static_cast<int>(std::min<long long>(n_items, num_sms()));
    // MMA rows: 64 when the tile's G x rows fit, else 128.  With 64 rows and
    // tile tables that fit beside two warpgroups' buffers, two items per SM
    // are in flight (attn_pp_kernel); otherwise one (attn_tc_kernel).
    const size_t pp_smem = pp_smem_bytes(n_tiles, W);
    int st;
    if (P.tile_rows * P.G <= 64 && pp_smem <= kPPSmemMax)
        st = launch_pdl(attn_pp_kernel, dim3(static_cast<unsigned>(grid)), dim3(kPPThreads), pp_smem, s, tk, tv,
                        tk2, tv2, tq, P);
    else if (P.tile_rows * P.G <= 64)
        st = launch_pdl(attn_tc_kernel<64>, dim3(static_cast<unsigned>(grid)), dim3(ATTN_THREADS),
                        tc_smem_bytes<64>(), s, tk, tv, tk2, tv2, P);
    else
        st = launch_pdl(attn_tc_kernel<128>, dim3(static_cast<unsigned>(grid)), dim3(ATTN_THREADS),
                        tc_smem_bytes<128>(), s, tk, tv, tk2, tv2, P);
    if (st != BIV_OK) return st;
    const long long n_pairs = static_cast<long long>(W) * Hq;
    const long long cgrid = std::min<long long>((n_pairs + 7) / 8, static_cast<long long>(num_sms()) * combine_per_sm);
    return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>(cgrid)), dim3(256), combine_smem_bytes(W, Hq, P.s_max, static_cast<int>(cgrid) * 8), s,
                      P, static_cast<__nv_bfloat16*>(o));
}

extern "C" int biv_rope_qk(const void* qkv, void* q_out, void* k_out, const int32_t* row_pos, int W, int Hq,
                           int Hkv, int hd, float theta, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || Hq <= 0 || Hkv < 0 || hd <= 0 || hd % 2 != 0 || hd > 256) return BIV_ERR_SHAPE;
    if (!(theta > 1.0f) || !std::isfinite(theta)) return BIV_ERR_VALUE;
    if (W == 0) return BIV_OK;
    if (!qkv || !q_out || !row_pos || (Hkv > 0 && !k_out)) return BIV_ERR_NULL;
    const long long total = static_cast<long long>(W) * (Hq + Hkv) * (hd / 2);
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 8192));
    return launch_pdl(rope_kernel, dim3(blocks), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(q_out),
                      static_cast<__nv_bfloat16*>(k_out), row_pos, W, Hq, Hkv, hd, theta);
}

extern "C" int biv_rope_kv_write(const void* qkv, void* q_out, void* k_cache, void* v_cache,
                                 const int32_t* row_slot, const int32_t* row_pos, const int32_t* rows_keep, int W,
                                 int K, int Hq, int Hkv, int hd, int n_slots, int max_len, float theta,
                                 biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || K < 1 || Hq <= 0 || Hkv <= 0 || hd <= 0 || hd % 8 != 0 || hd > 256 || n_slots <= 0 ||
        max_len <= 0)
        return BIV_ERR_SHAPE;
    if (W % K != 0) return BIV_ERR_SHAPE;
    if (!(theta > 1.0f) || !std::isfinite(theta)) return BIV_ERR_VALUE;
    if (W == 0) return BIV_OK;
    if (!qkv || !q_out || !k_cache || !v_cache || !row_slot || !row_pos) return BIV_ERR_NULL;
    if (!aligned16(qkv) || !aligned16(q_out) || !aligned16(k_cache) || !aligned16(v_cache)) return BIV_ERR_ALIGN;
    return launch_pdl(rope_kv_write_kernel, dim3(W), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(q_out),
                      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), row_slot, row_pos,
                      rows_keep, K, Hq, Hkv, hd, n_slots, max_len, theta);
}

extern "C" int biv_kv_overwrite(void* k_cache, void* v_cache, const void* k_new, long long k_stride,
                                const void* v_new, long long v_stride, const int32_t* row_slot,
                                const int32_t* row_pos, const int32_t* rows_keep, int W, int K, int Hkv, int hd,
                                int n_slots, int max_len, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || K < 1 || Hkv <= 0 || hd <= 0 || n_slots <= 0 || max_len <= 0) return BIV_ERR_SHAPE;
    const long long row = static_cast<long long>(Hkv) * hd;
    if (hd % 8 != 0 || k_stride % 8 != 0 || v_stride % 8 != 0 || k_stride < row || v_stride < row)
        return BIV_ERR_SHAPE;
    if (W % K != 0) return BIV_ERR_SHAPE;
    if (W == 0) return BIV_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !row_slot || !row_pos) return BIV_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new)) return BIV_ERR_ALIGN;
    return launch_pdl(kv_overwrite_kernel, dim3(W), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache),
                      static_cast<const __nv_bfloat16*>(k_new), k_stride, static_cast<const __nv_bfloat16*>(v_new),
                      v_stride, row_slot, row_pos, rows_keep, K, Hkv, hd, n_slots, max_len);
}

// ------------------------------------------------ no-alloc attention variant
// For callers that may not allocate device memory (an allocator owned by a
// host runtime, a plugin with no allocator handle): the attention partials
// live in this fixed array instead of a caller workspace.  It is device
// memory of the loaded module, BIV_NOALLOC_SCRATCH_BYTES per GPU, kept until
// the process exits.  In host code `g_attn_scratch` is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress, looked up once
// per device with that device current.
namespace biv {
namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[BIV_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr with
// *status set.
void* attn_scratch(int* status) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *status = cuda_status(e);
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *status = BIV_ERR_DEVICE;
        return nullptr;
    }
    std::lock_guard<std::mutex> g(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *status = cuda_status(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    *status = BIV_OK;
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace biv

extern "C" int biv_decode_attn_fixedsplit_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* row_slot, const int32_t* row_pos, void* o, int W,
                                                  int rows_per_group, int Hq, int Hkv, int hd, int n_slots,
                                                  int max_len, int kv_split, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || Hq <= 0 || Hkv <= 0 || n_slots <= 0 || max_len <= 0 || rows_per_group <= 0)
        return BIV_ERR_SHAPE;
    if (hd != HD || kv_split != SPLIT) return BIV_ERR_UNSUPPORTED;
    if (W == 0) return BIV_OK;
    if (biv_decode_attn_workspace_size(W, Hq, max_len) > BIV_NOALLOC_SCRATCH_BYTES) return BIV_ERR_SCRATCH;
    int st = BIV_OK;
    void* scratch = attn_scratch(&st);
    if (!scratch) return st;
    return biv_decode_attn_fixedsplit(q, k_cache, v_cache, row_slot, row_pos, o, W, rows_per_group, Hq, Hkv, hd,
                                      n_slots, max_len, kv_split, scratch, BIV_NOALLOC_SCRATCH_BYTES, stream);
}
