// Fixed-split decode attention, RoPE and the verifier's KV overwrite.
//
// [DVR] para 1: batch-invariant attention uses a fixed KV-split size with no
// adaptation to sequence length or GPU load.  [DVR] para 3: the verifier
// overwrites the fast path's cache rows with its own values before they are
// attended to.  [GUIDE] GQA tile rule: the G query heads that share a KV head,
// times the verified rows of one request, fill one 128-row MMA tile
// (G * (1 + D) <= 128).
//
// Phase 1, one CTA per (row tile, KV head, split of 256 absolute positions):
// the tile holds up to 128/G consecutive rows of one request times its G
// query heads.  K and V of the split are staged in shared memory once
// (cp.async, XOR-swizzled 16-byte chunks) and every row of the tile reuses
// them.  Each compute warp owns 16 tile rows; per 64-key chunk it forms
// S = Q K^T with bf16 mma.sync (fp32 accumulate), masks keys beyond the
// row's own position with a select, and updates an online softmax in a
// fixed order.  The split's partial (max, sum, unnormalised output) goes to
// the caller's workspace.  Phase 2 combines the splits 0..p/256 of each
// (row, head) in increasing order.  Nothing in a row's arithmetic depends on
// the other rows of the tile or the batch: masked keys contribute exact
// zeros and chunks beyond a row's position leave its state unchanged.
//
// The contraction per split is tiny (16..128 rows x 256 keys x 128), so the
// kernel is bound by reading K and V from HBM, not by the tensor pipe;
// mma.sync is ample here.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "biv_common.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_attn_err)

constexpr int HD = BIV_HEAD_DIM;        // 128
constexpr int SPLIT = BIV_KV_SPLIT;     // 256
constexpr int CHUNK = 64;               // keys per online-softmax step
constexpr int ROWB = HD * 2;            // 256 bytes per K/V/Q row in shared memory
constexpr int ATTN_THREADS = 256;
constexpr int kPartialBytes = (4 * 16 * HD + 2 * 4 * 16) * 4;   // chunk partials of one 16-row block

// Byte offset of (row, 16-byte chunk) in a swizzled [rows][128] bf16 tile.
BIV_DEV uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * ROWB + ((chunk ^ (row & 7)) << 4));
}

// K or V of one split as TMA writes it: per 64-key chunk a [2 halves][64 keys]
// [128 B] image with 128-byte swizzle (16-byte piece j of a 128-byte row r is
// stored at piece j ^ (r % 8)).  Byte offset of (key, 16-byte piece c of the
// 256-byte row).
constexpr int kKvChunkBytes = CHUNK * ROWB;   // 16 KiB
BIV_DEV uint32_t swz_kv(int key, int c) {
    const int r = key & (CHUNK - 1);
    return static_cast<uint32_t>((key >> 6) * kKvChunkBytes + (c >> 3) * (kKvChunkBytes / 2) + r * 128 +
                                 (((c & 7) ^ (r & 7)) << 4));
}

BIV_DEV void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
BIV_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
BIV_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

BIV_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
BIV_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32.
BIV_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                            uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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

// Per-tile tables in shared memory, built by all threads of the CTA: the
// largest usable position of each tile (-1: none), its first row's cache
// slot, and the exclusive prefix sums of its live work items
// (Hkv * (tmax / SPLIT + 1) each); s_pref[kMaxTilesSmem] is the live total.
// Returns whether the tables cover every tile (else callers fall back to all
// (split, KV head, tile) triples with the dead ones skipped).
BIV_DEV bool build_tile_tables(const AttnParams& P, int* s_tmax, int* s_pref, int* s_slot0, int* s_wsum) {
    const int n_tiles = P.n_tiles;
    // Largest usable position of each tile, one thread per row (independent
    // loads); tiles past the table are scanned where they are processed.
    for (int t = threadIdx.x; t < min(n_tiles, kMaxTilesSmem); t += ATTN_THREADS) s_tmax[t] = -1;
    __syncthreads();
    for (int w = threadIdx.x; w < P.W; w += ATTN_THREADS) {
        const int group = w / P.rows_per_group;
        const int sub = (w - group * P.rows_per_group) / P.tile_rows;
        const int t = group * P.tiles_per_group + sub;
        if (t >= kMaxTilesSmem) break;                       // rows only grow the tile index
        const int row0 = group * P.rows_per_group + sub * P.tile_rows;
        const int slot0 = P.row_slot[row0];
        if (w == row0) s_slot0[t] = slot0;
        if (slot0 < 0 || slot0 >= P.n_slots) {
            if (w == row0 && blockIdx.x == 0) atomicOr(&g_attn_err, BIV_DEVERR_INDEX);
            continue;
        }
        const int s = P.row_slot[w], p = P.row_pos[w];
        if (s == slot0 && p >= 0 && p < P.max_len) atomicMax(&s_tmax[t], p);
    }
    __syncthreads();
    // Live work items: tile t has Hkv * (s_tmax[t] / SPLIT + 1) of them (none
    // if no row is usable); s_pref holds their exclusive prefix sums, so the
    // CTAs can deal out exactly the live items, consecutive ones to
    // consecutive CTAs.  Tables too large for shared memory fall back to all
    // (split, KV head, tile) triples with the dead ones skipped.
    const bool live_mode = n_tiles <= kMaxTilesSmem;
    if (live_mode) {
        // thread i scans tiles [i * per, (i + 1) * per); warp and block prefix
        const int per = (n_tiles + ATTN_THREADS - 1) / ATTN_THREADS;
        const int t0 = min(static_cast<int>(threadIdx.x) * per, n_tiles);
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
        if (lane == 31) s_wsum[warp] = inc;
        __syncthreads();
        int base = inc - sum;
        for (int w = 0; w < warp; ++w) base += s_wsum[w];
        for (int t = t0; t < t1; ++t) {
            s_pref[t] = base;
            base += s_tmax[t] >= 0 ? P.Hkv * (s_tmax[t] / SPLIT + 1) : 0;
        }
        if (threadIdx.x == ATTN_THREADS - 1) s_pref[kMaxTilesSmem] = base;   // the live total
        __syncthreads();
    }
    return live_mode;
}

__global__ void __launch_bounds__(ATTN_THREADS)
attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const AttnParams P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    __shared__ int s_pos[BIV_ATTN_TILE];
    __shared__ __align__(8) uint64_t kv_bar[SPLIT / CHUNK];    // one per 64-key chunk (K and V)
    __shared__ int abort_flag;
    __shared__ int s_tmax[kMaxTilesSmem];                      // largest row position per tile
    __shared__ int s_pref[kMaxTilesSmem + 1];                  // live items before each tile; [kMax] = total
    __shared__ int s_slot0[kMaxTilesSmem];                     // cache slot of each tile's first row
    __shared__ int s_wsum[ATTN_THREADS / 32];

    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int c = 0; c < SPLIT / CHUNK; ++c) mbar_init(&kv_bar[c], 1);
        fence_mbar_init();
    }
    const int n_tiles = P.n_tiles;
    const bool live_mode = build_tile_tables(P, s_tmax, s_pref, s_slot0, s_wsum);
    uint32_t kv_parity = 0;                     // bit c: phase parity of chunk barrier c
    const long long n_work =
        live_mode ? s_pref[kMaxTilesSmem] : static_cast<long long>(P.s_max) * P.Hkv * n_tiles;
#pragma unroll 1
    for (long long item = blockIdx.x; item < n_work; item += gridDim.x) {
    int tile, kvh, split;
    if (live_mode) {
        // the tile whose prefix range holds the item: the last t with s_pref[t] <= item
        int lo = 0, hi = n_tiles - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pref[mid] <= item) lo = mid; else hi = mid - 1;
        }
        tile = lo;
        const int r = static_cast<int>(item - s_pref[lo]);
        kvh = r % P.Hkv;
        split = r / P.Hkv;
    } else {
        tile = static_cast<int>(item % n_tiles);
        const long long rest = item / n_tiles;
        kvh = static_cast<int>(rest % P.Hkv);
        split = static_cast<int>(rest / P.Hkv);
    }
    const int key0 = split * SPLIT;
    const int maxpos = tile < kMaxTilesSmem ? s_tmax[tile] : tile_maxpos(P, tile);
    if (maxpos < key0) continue;                // no row of the tile reaches this split
    int row0, nr;
    tile_rows_of(P, tile, row0, nr);
    const int T = nr * P.G;                     // live tile rows (row-major over (row, head))
    const int T16 = (T + 15) & ~15;

    // a processed tile's first row has a usable slot (else the tile has no items)
    const int slot0 = live_mode ? s_slot0[tile] : P.row_slot[row0];
    const int n_keys = min(SPLIT, maxpos + 1 - key0);
    const int n_chunks = (n_keys + CHUNK - 1) / CHUNK;

    uint8_t* sQ = smem;                         // [T16][HD], 256-B rows, swz()
    uint8_t* sK = smem + ((T16 * ROWB + 1023) & ~1023);   // [4 chunks] TMA images, swz_kv()
    uint8_t* sV = sK + SPLIT * ROWB;
    const uint32_t uQ = smem_u32(sQ), uK = smem_u32(sK), uV = smem_u32(sV);

    // ---- K/V of the split first: one TMA box per 64-key chunk and matrix,
    // each chunk completing on its own barrier; then the rows' positions and
    // Q (zero rows >= T) with cp.async.
    if (threadIdx.x == 0) {
        fence_proxy_async_smem();               // earlier generic writes to this memory come first
        const int kv_row = (slot0 * P.Hkv + kvh) * P.max_len + key0;
        for (int c = 0; c < n_chunks; ++c) {
            mbar_arrive_expect_tx(&kv_bar[c], 2u * kKvChunkBytes);
            tma_load_3d(sK + c * kKvChunkBytes, &tmK, &kv_bar[c], 0, kv_row + c * CHUNK, 0, policy_evict_first());
            tma_load_3d(sV + c * kKvChunkBytes, &tmV, &kv_bar[c], 0, kv_row + c * CHUNK, 0, policy_evict_first());
        }
    }
    if (threadIdx.x < nr) {
        const int w = row0 + threadIdx.x;
        int p = -1;
        if (row_ok(P, w, slot0)) p = P.row_pos[w];
        s_pos[threadIdx.x] = p;
    }
    for (int idx = threadIdx.x; idx < T16 * 16; idx += ATTN_THREADS) {
        const int t = idx >> 4, c = idx & 15;
        if (t < T) {
            const int i = t / P.G, g = t - i * P.G;
            const __nv_bfloat16* src =
                P.q + (static_cast<long long>(row0 + i) * P.Hq + kvh * P.G + g) * HD + c * 8;
            cp_async16(uQ + swz(t, c), src);
        } else {
            *reinterpret_cast<uint4*>(sQ + swz(t, c)) = make_uint4(0, 0, 0, 0);
        }
    }
    cp_async_commit();

    // ---- per block of 16 tile rows, warp w takes 64-key chunk w / 2 and head
    // dims [64 (w % 2), 64 (w % 2) + 64): S = Q K^T over the chunk, its softmax,
    // O = P V for its dims.  The four chunk partials are merged in increasing
    // chunk order.  Every row's arithmetic is the same whatever else is in
    // the tile.
    cp_async_wait<0>();
    __syncthreads();                            // Q (and the barrier init) visible to all
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;     // mma fragment coordinates
    const int ch = warp >> 1, hh = warp & 1;
    bool have = false;                          // this warp's chunk landed
    if (ch < n_chunks) {
        have = mbar_wait(&kv_bar[ch], (kv_parity >> ch) & 1u, &abort_flag, &g_attn_err);
        // Keys past the last one any row of the tile reads may hold anything
        // (they are read in whole 64-key boxes): zero this warp's half of V there,
        // so a masked score (p = 0) never meets a NaN.  K needs nothing: its
        // scores are replaced by -inf with a select.
        const int nk = n_keys - ch * CHUNK;
        if (have && nk < CHUNK) {
            for (int idx = lane; idx < (CHUNK - nk) * 8; idx += 32) {
                const int key = ch * CHUNK + nk + (idx >> 3), c = hh * 8 + (idx & 7);
                *reinterpret_cast<uint4*>(sV + swz_kv(key, c)) = make_uint4(0, 0, 0, 0);
            }
        }
        __syncwarp();
    }
    float* sPO = reinterpret_cast<float*>(sV + SPLIT * ROWB);    // [4 chunks][16 rows][HD]
    float* sPM = sPO + 4 * 16 * HD;                              // [4][16] chunk maxima (log2 units)
    float* sPL = sPM + 4 * 16;                                   // [4][16] chunk weight sums

#pragma unroll 1
    for (int rb = 0; rb < T16 / 16; ++rb) {
        const int trow_a = rb * 16 + gq, trow_b = trow_a + 8;
        const int pos_a = trow_a < T ? s_pos[trow_a / P.G] : -1;
        const int pos_b = trow_b < T ? s_pos[trow_b / P.G] : -1;
        float o[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
        float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
        if (have) {
            // ---- S = Q K^T for 16 rows x 64 keys
            float sc[8][4];
#pragma unroll
            for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.0f;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(uQ + swz(rb * 16 + (lane & 15), kk * 2 + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    const int j = lane >> 3;
                    const int key = ch * CHUNK + np * 16 + (j >> 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(uK + swz_kv(key, kk * 2 + (j & 1)), b0, b1, b2, b3);
                    mma_bf16_16816(sc[2 * np], a0, a1, a2, a3, b0, b1);
                    mma_bf16_16816(sc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                }
            }
            // ---- mask (select, never multiply), scale into log2 units, chunk max
            const int kbase = key0 + ch * CHUNK + cq * 2;
            float cmax_a = -INFINITY, cmax_b = -INFINITY;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = kbase + n * 8 + e;
                    sc[n][e] = key <= pos_a ? sc[n][e] * P.scale_log2 : -INFINITY;
                    sc[n][2 + e] = key <= pos_b ? sc[n][2 + e] * P.scale_log2 : -INFINITY;
                    cmax_a = fmaxf(cmax_a, sc[n][e]);
                    cmax_b = fmaxf(cmax_b, sc[n][2 + e]);
                }
            }
            cmax_a = fmaxf(cmax_a, __shfl_xor_sync(0xffffffffu, cmax_a, 1));
            cmax_a = fmaxf(cmax_a, __shfl_xor_sync(0xffffffffu, cmax_a, 2));
            cmax_b = fmaxf(cmax_b, __shfl_xor_sync(0xffffffffu, cmax_b, 1));
            cmax_b = fmaxf(cmax_b, __shfl_xor_sync(0xffffffffu, cmax_b, 2));
            const float mu_a = cmax_a == -INFINITY ? 0.0f : cmax_a;   // a row with no key in the chunk
            const float mu_b = cmax_b == -INFINITY ? 0.0f : cmax_b;
            m_a = cmax_a;
            m_b = cmax_b;
#pragma unroll
            for (int n = 0; n < 8; ++n) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sc[n][e] = exp2f(sc[n][e] - mu_a);
                    sc[n][2 + e] = exp2f(sc[n][2 + e] - mu_b);
                    l_a += sc[n][e];
                    l_b += sc[n][2 + e];
                }
            }
            // ---- O = P V for this warp's 64 dims (P from the S accumulators)
#pragma unroll
            for (int kk = 0; kk < CHUNK / 16; ++kk) {
                const uint32_t p0 = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
                const uint32_t p1 = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
                const uint32_t p2 = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                const uint32_t p3 = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
                for (int nd = 0; nd < 4; ++nd) {
                    const int j = lane >> 3;
                    const int key = ch * CHUNK + kk * 16 + (j & 1) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(uV + swz_kv(key, (hh * 4 + nd) * 2 + (j >> 1)), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * nd], p0, p1, p2, p3, b0, b1);
                    mma_bf16_16816(o[2 * nd + 1], p0, p1, p2, p3, b2, b3);
                }
            }
            // row sums across the quad (fixed order)
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
        }
        // ---- the chunk partial into shared memory
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int d = hh * 64 + n * 8 + cq * 2;
            *reinterpret_cast<float2*>(sPO + (ch * 16 + gq) * HD + d) = make_float2(o[n][0], o[n][1]);
            *reinterpret_cast<float2*>(sPO + (ch * 16 + gq + 8) * HD + d) = make_float2(o[n][2], o[n][3]);
        }
        if (hh == 0 && cq == 0) {
            sPM[ch * 16 + gq] = m_a;
            sPM[ch * 16 + gq + 8] = m_b;
            sPL[ch * 16 + gq] = l_a;
            sPL[ch * 16 + gq + 8] = l_b;
        }
        __syncthreads();
        // ---- merge the four chunks (increasing order), write the split's partial
        {
            const int r = threadIdx.x >> 4, d0 = (threadIdx.x & 15) * 8;
            const int trow = rb * 16 + r;
            const int pos = trow < T ? s_pos[trow / P.G] : -1;
            if (pos >= key0) {
                float M = sPM[r];
#pragma unroll
                for (int c = 1; c < 4; ++c) M = fmaxf(M, sPM[c * 16 + r]);
                float L = 0.0f;
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float mc = sPM[c * 16 + r];
                    const float wc = mc == -INFINITY ? 0.0f : exp2f(mc - M);
                    L += wc * sPL[c * 16 + r];
                    const float4 u0 = *reinterpret_cast<const float4*>(sPO + (c * 16 + r) * HD + d0);
                    const float4 u1 = *reinterpret_cast<const float4*>(sPO + (c * 16 + r) * HD + d0 + 4);
                    acc[0] += wc * u0.x; acc[1] += wc * u0.y; acc[2] += wc * u0.z; acc[3] += wc * u0.w;
                    acc[4] += wc * u1.x; acc[5] += wc * u1.y; acc[6] += wc * u1.z; acc[7] += wc * u1.w;
                }
                const int i = trow / P.G, g = trow - i * P.G;
                const long long ph = (static_cast<long long>(row0 + i) * P.Hq + kvh * P.G + g) * P.s_max + split;
                float* dst = P.ws_o + ph * HD + d0;
                *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                if (d0 == 0) {
                    P.ws_m[ph] = M;
                    P.ws_l[ph] = L;
                }
            }
        }
        __syncthreads();      // the partial buffers are reused by the next row block
    }
    if (threadIdx.x == 0 && abort_flag)
        for (int c = 0; c < n_chunks; ++c) mbar_wait_drain(&kv_bar[c], (kv_parity >> c) & 1u);   // land first
    kv_parity ^= (1u << n_chunks) - 1u;
    if (abort_flag) break;
    }
}

// One warp per (row, head): combine splits 0 .. pos/256 of the row.  Lane s
// holds split s (32 at a time); the maximum and the weight sum are reduced
// with a fixed xor butterfly, the outputs are summed in increasing split
// order.  All loads of a group of splits are independent, so they overlap.
__global__ void __launch_bounds__(256)
attn_combine_kernel(const AttnParams P, __nv_bfloat16* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    const long long pair = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (pair >= static_cast<long long>(P.W) * P.Hq) return;
    const int w = static_cast<int>(pair / P.Hq);
    const int grp0 = (w / P.rows_per_group) * P.rows_per_group;
    const int slot = P.row_slot[w], p = P.row_pos[w], slot0 = P.row_slot[grp0];
    __nv_bfloat16* dst = out + pair * HD + lane * 4;
    if (slot < 0 || slot >= P.n_slots || p < 0 || p >= P.max_len || slot != slot0) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
        return;
    }
    const int ns = p / SPLIT + 1;
    const long long base = pair * P.s_max;
    // Row maximum over all splits.
    float M = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 32) {
        float m = (s0 + lane < ns) ? P.ws_m[base + s0 + lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        M = fmaxf(M, m);
    }
    float L = 0.0f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += 32) {
        const int s = s0 + lane;
        const float wgt = (s < ns) ? exp2f(P.ws_m[base + s] - M) : 0.0f;
        float lw = (s < ns) ? wgt * P.ws_l[base + s] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        L += lw;
        const int cnt = min(32, ns - s0);
        const float4* src = reinterpret_cast<const float4*>(P.ws_o + (base + s0) * HD) + lane;
#pragma unroll 4
        for (int j = 0; j < cnt; ++j) {
            const float wj = __shfl_sync(0xffffffffu, wgt, j);
            const float4 v = src[static_cast<long long>(j) * (HD / 4)];
            acc.x += wj * v.x;
            acc.y += wj * v.y;
            acc.z += wj * v.z;
            acc.w += wj * v.w;
        }
    }
    const float inv = 1.0f / L;
    uint2 r;
    r.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    r.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = r;
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
    return static_cast<size_t>(pairs) * (HD + 2) * sizeof(float);
}

extern "C" int biv_gqa_max_drafts(int G, int tile) {
    if (G <= 0 || G > tile) return -1;
    return tile / G - 1;
}

extern "C" int biv_decode_attn_fixedsplit(const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* row_slot, const int32_t* row_pos, void* o, int W,
                                          int rows_per_group, int Hq, int Hkv, int hd, int n_slots, int max_len,
                                          int kv_split, void* workspace, size_t ws_bytes, biv_stream_t stream) {
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
    P.ws_o = static_cast<float*>(workspace);
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
    const int T16max = ((P.tile_rows * P.G + 15) / 16) * 16;
    const size_t smem = 1024 + ((static_cast<size_t>(T16max) * ROWB + 1023) & ~static_cast<size_t>(1023)) +
                        2 * SPLIT * ROWB + kPartialBytes;
    // K and V caches as TMA sees them: [2 halves of a row][n_slots*Hkv*max_len rows][64 elements]
    CUtensorMap tk, tv;
    {
        EncodeTiledFn enc = encode_fn();
        if (!enc) {
            set_cuda_error(cudaErrorNotSupported);
            return BIV_ERR_CUDA;
        }
        cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(n_slots) * Hkv * max_len, 2};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(ROWB), 128};
        cuuint32_t box[3] = {64, CHUNK, 2};
        cuuint32_t es[3] = {1, 1, 1};
        const void* bases[2] = {k_cache, v_cache};
        CUtensorMap* maps[2] = {&tk, &tv};
        for (int i = 0; i < 2; ++i) {
            if (enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(bases[i]), dims, strides, box,
                    es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
                set_cuda_error(cudaErrorInvalidValue);
                return BIV_ERR_CUDA;
            }
        }
    }

    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(attn_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             1024 + BIV_ATTN_TILE * ROWB + 2 * SPLIT * ROWB + kPartialBytes);
        if (e != cudaSuccess) return cuda_status(e);
        configured_device = dev;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long n_items = static_cast<long long>(s_max) * Hkv * n_tiles;
    const int grid = static_cast<int>(std::min<long long>(n_items, num_sms()));
    int st = launch_pdl(attn_split_kernel, dim3(static_cast<unsigned>(grid)), dim3(ATTN_THREADS), smem, s, tk, tv, P);
    if (st != BIV_OK) return st;
    const long long n_pairs = static_cast<long long>(W) * Hq;
    return launch_pdl(attn_combine_kernel, dim3(static_cast<unsigned>((n_pairs + 7) / 8)), dim3(256), 0, s, P,
                      static_cast<__nv_bfloat16*>(o));
}

extern "C" int biv_rope_qk(const void* qkv, void* q_out, void* k_out, const int32_t* row_pos, int W, int Hq,
                           int Hkv, int hd, float theta, biv_stream_t stream) {
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

constexpr int kMaxDevices = 64;
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
