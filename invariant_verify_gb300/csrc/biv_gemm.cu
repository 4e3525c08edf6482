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
// Kernel layout (320 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: per stage one box of A [a_rows x KS*64] and one of
//               B [BN x KS*64] (3-D tensor maps: KS k-blocks of 64 per box; the
//               TMA unit spends a fixed ~275 ns per box whatever its size, so
//               weight-streaming tiles take as many k-blocks per box as two
//               stages allow), 128-byte swizzle, mbarrier transaction
//               counts.  For M <= 128 only the real rows of A are copied
//               (a_rows = M rounded up to 8) and packed back to back; the
//               MMA still reads 128 rows per k-block, and the rows past
//               a_rows hold unrelated data -- harmless, because each row of the
//               product depends only on its own row of A and rows >= M are
//               never stored.
//   warp 1      TMEM allocator + MMA issuer (one elected lane); commits free smem
//               stages and publish finished accumulators.
//   warps 2..9  epilogue, two warps per TMEM lane quarter (each takes half of
//               a tile's columns): tcgen05.ld, convert, store.
// Two accumulators in TMEM let the epilogue of tile i overlap the MMAs of
// tile i + 1.  Launched with programmatic dependent launch: barrier set-up
// and TMEM allocation overlap the previous kernel.  Every wait is
// bounded (2 s); on time-out the kernel raises BIV_DEVERR_TIMEOUT, drains its
// in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "biv_common.cuh"
#include "biv_gumbel.cuh"

namespace biv {
namespace {

BIV_DEFINE_ERR_WORD(g_gemm_err)

constexpr int kBM = 128;
constexpr int kBK = 64;                       // 64 bf16 = one 128-byte swizzle row
constexpr int kRowBytes = kBK * 2;            // one 64-wide k-block row: 128 B
constexpr int kTailSlack = kBM * kRowBytes;   // the MMA may read 128 A rows past the last stage
constexpr int kMaxStages = 24;
constexpr int kBarBytes = 512;
constexpr int kWave = 152;                    // CTAs of one wave on a 152-SM part
constexpr int kPairWave = kWave / 2;          // 2-CTA clusters of one wave
constexpr int kMaxSmem = 227 * 1024;          // opt-in shared memory per block

struct GemmArgs {
    int M, N, K;
    int BN;          // tile width (multiple of 16, 16..256)
    int KS;          // 64-wide k-blocks per stage (one TMA box each for A and B)
    int KB;          // k-blocks in K
    int three_d;     // 3-D tensor maps (K % 64 == 0), else 2-D with KS = 1
    int stages;      // ring depth
    int first1;      // the first stage of every tile is one k-block (3-D maps tmA1/tmB1), so the
                     // MMAs start as soon as it lands; the others hold KS k-blocks
    int m64;         // one row tile of at most 64 rows: M = 64 MMAs
    int a_rows;      // rows of A copied per k-block (multiple of 8, <= 128)
    uint32_t idesc;  // tcgen05 instruction descriptor for M=128, N=BN
    uint32_t tmem_cols;
    // Narrow tail (CTA pairs, fused selection): column tiles [0, nt_full) are
    // BN wide and the rest bn_tail wide (tensor map tmB1, descriptor
    // idesc_tail), so that the last, partial wave of full tiles becomes one
    // wave of narrower tiles.  bn_tail = 0: every column tile is BN wide.
    int nt_full;
    int bn_tail;
    uint32_t idesc_tail;
};

// Tile t of the persistent schedule (row tiles fastest): its row tile, first
// column, width and column-tile index (the selection's winner slot).
struct TileAt {
    int m_blk, col0, bn, slot;
};

BIV_DEV TileAt tile_at(const GemmArgs& g, int t, int m_tiles) {
    const int full = g.nt_full * m_tiles;
    if (g.bn_tail == 0 || t < full) {
        const int nb = t / m_tiles;
        return TileAt{t - nb * m_tiles, nb * g.BN, g.BN, nb};
    }
    const int u = t - full, nb = u / m_tiles;
    return TileAt{u - nb * m_tiles, g.nt_full * g.BN + nb * g.bn_tail, g.bn_tail, g.nt_full + nb};
}

// Column tiles of the schedule (full and narrow).
BIV_DEV int column_tiles(const GemmArgs& g) {
    return g.bn_tail == 0 ? (g.N + g.BN - 1) / g.BN
                          : g.nt_full + (g.N - g.nt_full * g.BN + g.bn_tail - 1) / g.bn_tail;
}

inline int stage_bytes(int KS, int a_rows, int BN) { return KS * (a_rows + BN) * kRowBytes; }

// k-blocks [kb0, kb0 + nkb) of stage sb of a tile.
BIV_DEV void stage_range(const GemmArgs& g, int sb, int& kb0, int& nkb) {
    if (g.first1) {
        kb0 = sb == 0 ? 0 : 1 + (sb - 1) * g.KS;
        nkb = sb == 0 ? 1 : min(g.KS, g.KB - kb0);
    } else {
        kb0 = sb * g.KS;
        nkb = min(g.KS, g.KB - kb0);
    }
}

// Selection fused into the LM-head epilogue (EPI 3): every tile-row's Gumbel
// winner, packed as (order(key) << 32 | ~v), goes to cand[row * n_cols + c] for
// column tile c (n_cols column tiles in all, see TailPlan).
struct SelectArgs {
    const uint32_t* row_req;
    const int32_t* row_pos;
    unsigned long long* cand;
    uint32_t seed_lo, seed_hi;
    float invT;
    int greedy;
};

BIV_DEV uint32_t pick_word(const U4& w, uint32_t j) {
    return j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
}

// Epilogue threads per CTA: 256 (warps 2-9: two per TMEM lane quarter, each
// taking half of a tile's columns, so two warps share every SM sub-partition's
// issue slots).  With one warp per quarter the 2-layer W = 64 step was 0.7 us
// slower (its GEMMs have a single tile per CTA, so every epilogue is on the
// path); at W = 1024 the exposed last-tile epilogues are bound by their
// scattered stores, not by issue, and did not change.
template <int EPI>
__host__ __device__ constexpr int epi_threads() { return 256; }

// Column range [cb, ce) of a tile of width bn that warp set `eset` (0: warps
// 2-5, 1: warps 6-9) takes, in whole units of `unit` columns.
BIV_DEV void eset_columns(int bn, int unit, int eset, int& cb, int& ce) {
    const int units = (bn + unit - 1) / unit, h = (units + 1) / 2;
    cb = eset ? h * unit : 0;
    ce = eset ? bn : min(bn, h * unit);
}

template <int NT>
BIV_DEV void epilogue_bar() {
    if constexpr (NT == 256)
        asm volatile("bar.sync 1, 256;" ::: "memory");
    else
        asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Barrier over the NT epilogue threads that also ANDs a flag across them, so
// that a failed wait makes all of them leave the tile loop together.
template <int NT>
BIV_DEV bool epilogue_all(bool v) {
    uint32_t r;
    if constexpr (NT == 256)
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, 256, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}\n"
            : "=r"(r)
            : "r"(static_cast<uint32_t>(v))
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 1, 128, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}\n"
            : "=r"(r)
            : "r"(static_cast<uint32_t>(v))
            : "memory");
    return r != 0;
}

// Noise buckets (EPI 3): bucket b of a Philox word w is its top 12 bits,
// b = w >> 20 (2^11 consecutive uniform indices).  The noise is a
// non-decreasing function of the uniform index, so the noise at a bucket's
// top word bounds every noise in the bucket.  T[b] is that bound for the top
// 256 buckets (noise above 2.7, where the winners are decided) and the bound
// of the enclosing 8-bit bucket (top byte b >> 4) below them.
constexpr int kBucketBits = 12;
constexpr int kBuckets = 1 << kBucketBits;
// RoPE + KV-write epilogue (EPI 4) of the QKV projection: the weight rows are
// rearranged (biv_rope_pack_qkv_weights) so that every 16 output columns of
// the q and k part hold 8 rotation pairs of one head -- dims i0..i0+7 then
// i0+hd/2..i0+hd/2+7, i0 = 8 gq -- ordered frequency group first ([gq][head]
// [16]), and one thread rotates them from its own registers.  A tile's columns
// then span one or two frequency groups across many heads, so a thread takes
// the sines and cosines of its row once per group, not once per head.
struct RopeArgs {
    __nv_bfloat16* q_out;      // [M, Hq, hd]
    __nv_bfloat16* kc;         // [n_slots, Hkv, max_len, hd]
    __nv_bfloat16* vc;
    __nv_bfloat16* qkv_out;    // the unrotated projection in the original column order, or null
    const int32_t* row_slot;
    const int32_t* row_pos;
    const int32_t* rows_keep;  // [M / K] or null
    int Hq, Hkv, hd, n_slots, max_len, K;
    float theta;
};

// NP bf16 (NP / 2 packed pairs) in one vector store.
template <int NP>
BIV_DEV void st_bf16s(__nv_bfloat16* p, const uint32_t* v) {
    if constexpr (NP == 8)
        *reinterpret_cast<uint4*>(p) = make_uint4(v[0], v[1], v[2], v[3]);
    else
        *reinterpret_cast<uint2*>(p) = make_uint2(v[0], v[1]);
}

// The sines and cosines of one row's NP rotation pairs 8 gq + jb .. of
// frequency group gq, kept while consecutive column groups share gq.
template <int NP>
struct RopeAngles {
    int gq = -1;
    float sn[NP], cs[NP];
    BIV_DEV void at(int g, int jb, int pos, const float* inv_freq) {
        if (g == gq) return;
        gq = g;
#pragma unroll
        for (int j = 0; j < NP; ++j) rope_sincos(pos, inv_freq[8 * g + jb + j], sn[j], cs[j]);
    }
};

// One row's share of a 16-column group at output column col of the QKV tile:
// f1 holds the fp32 accumulators of group columns jb .. jb + NP - 1 (first
// halves of rotation pairs jb ..), f2 those of columns 8 + jb .. (their
// partners). q and k pairs are rotated at the row's position and stored to
// q_out or the k cache; v columns go to the v cache unrotated.
template <int NP>
BIV_DEV void qkv_group(const uint32_t* f1, const uint32_t* f2, int jb, int col, int row, int slot, int pos,
                       bool write_kv, const RopeArgs& rp, const float* inv_freq, RopeAngles<NP>& ang) {
    const int hd = rp.hd, half = hd / 2;
    const int qn = rp.Hq * hd, kn = rp.Hkv * hd;
    uint32_t a[NP / 2], b[NP / 2];                // bf16 pairs, as the plain GEMM stores them
#pragma unroll
    for (int e = 0; e < NP / 2; ++e) {
        a[e] = pack_bf16x2(__uint_as_float(f1[2 * e]), __uint_as_float(f1[2 * e + 1]));
        b[e] = pack_bf16x2(__uint_as_float(f2[2 * e]), __uint_as_float(f2[2 * e + 1]));
    }
    __nv_bfloat16* qkv_row = rp.qkv_out ? rp.qkv_out + static_cast<long long>(row) * (qn + 2 * kn) : nullptr;
    if (col < qn + kn) {
        const int nqk = rp.Hq + rp.Hkv;
        const int gi = col / 16, gq = gi / nqk, hh = gi - gq * nqk;
        const bool isq = hh < rp.Hq;
        const int h = isq ? hh : hh - rp.Hq, i0 = 8 * gq + jb;
        ang.at(gq, jb, pos, inv_freq);
        uint32_t o1[NP / 2], o2[NP / 2];
#pragma unroll
        for (int j = 0; j < NP; j += 2) {
            __nv_bfloat16 a0, a1, b0, b1;
            rope_rotate(bf16lo(a[j / 2]), bf16lo(b[j / 2]), ang.sn[j], ang.cs[j], a0, b0);
            rope_rotate(bf16hi(a[j / 2]), bf16hi(b[j / 2]), ang.sn[j + 1], ang.cs[j + 1], a1, b1);
            o1[j / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(a0)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(a1)) << 16);
            o2[j / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(b0)) |
                        (static_cast<uint32_t>(__bfloat16_as_ushort(b1)) << 16);
        }
        __nv_bfloat16* dst = nullptr;
        if (isq)
            dst = rp.q_out + (static_cast<long long>(row) * rp.Hq + h) * hd;
        else if (write_kv)
            dst = rp.kc + ((static_cast<long long>(slot) * rp.Hkv + h) * rp.max_len + pos) * hd;
        if (dst) {
            st_bf16s<NP>(dst + i0, o1);
            st_bf16s<NP>(dst + half + i0, o2);
        }
        if (qkv_row) {
            __nv_bfloat16* base = qkv_row + (isq ? 0 : qn) + h * hd;
            st_bf16s<NP>(base + i0, a);
            st_bf16s<NP>(base + half + i0, b);
        }
    } else {
        const int cc = col - qn - kn;
        const int h = cc / hd, d0 = cc % hd;
        if (write_kv) {
            __nv_bfloat16* dst = rp.vc + ((static_cast<long long>(slot) * rp.Hkv + h) * rp.max_len + pos) * hd + d0;
            st_bf16s<NP>(dst + jb, a);
            st_bf16s<NP>(dst + 8 + jb, b);
        }
        if (qkv_row) {
            __nv_bfloat16* base = qkv_row + qn + kn + cc;
            st_bf16s<NP>(base + jb, a);
            st_bf16s<NP>(base + 8 + jb, b);
        }
    }
}

constexpr int kNoiseTableBytes = kBuckets * 4 + 256 * 4;
constexpr int kExactBuckets = 256;
constexpr int kChunk = 32;                    // TMEM columns per load
constexpr int kMaxChunks = 256 / kChunk;

template <int NT>
BIV_DEV void fill_noise_table(float* ntab, float* t8) {
    const int e = static_cast<int>(threadIdx.x) - 64;            // 0..NT-1
    for (int b = e; b < 256; b += NT) t8[b] = gumbel_from_word((static_cast<uint32_t>(b) << 24) | 0x00ffffffu);
    for (int b = e; b < kExactBuckets; b += NT) {
        const uint32_t bb = static_cast<uint32_t>(kBuckets - kExactBuckets + b);
        ntab[bb] = gumbel_from_word((bb << (32 - kBucketBits)) | ((1u << (32 - kBucketBits)) - 1u));
    }
    epilogue_bar<NT>();
    for (int b = e; b < kBuckets - kExactBuckets; b += NT) ntab[b] = t8[b >> (kBucketBits - 8)];
}

// Buckets of one output tile, computed by the NT epilogue threads while the
// tile's MMAs run (the noise does not depend on the logits): for row r and
// group gq (entries v0 = n0 + 4 gq .. v0 + 3) bk[gq * RC + r] holds the four
// 16-bit buckets, entry j in bits [16 j, 16 j + 16) (group-major, so the 32
// rows of a warp read 32 consecutive words).
template <int NT>
BIV_DEV void tile_buckets(unsigned long long* bk, int RC, int rows, int BN, int n0, int N, int row0,
                          const SelectArgs& sel) {
    const int G4 = BN / 4;
    const int total = rows * G4;
    int gq = 0, r = static_cast<int>(threadIdx.x) - 64;
    while (r >= rows) { r -= rows; ++gq; }
    for (int idx = static_cast<int>(threadIdx.x) - 64; idx < total; idx += NT) {
        const uint32_t v0 = static_cast<uint32_t>(n0 + 4 * gq);
        unsigned long long packed = 0;
        if (v0 < static_cast<uint32_t>(N)) {
            const uint32_t req = sel.row_req[row0 + r];
            const uint32_t pos = static_cast<uint32_t>(sel.row_pos[row0 + r]) + 1u;
            const U4 w = philox4x32_10(v0 >> 2, pos, req, 0u, sel.seed_lo, sel.seed_hi);
            constexpr int sh = 32 - kBucketBits;
            packed = static_cast<unsigned long long>((w.x >> sh) | ((w.y >> sh) << 16)) |
                     (static_cast<unsigned long long>((w.z >> sh) | ((w.w >> sh) << 16)) << 32);
        }
        bk[gq * RC + r] = packed;
        r += NT;
        while (r >= rows) { r -= rows; ++gq; }
    }
}

// Bounds fl(fl(x * invT) + T[bucket]) of SEGW consecutive entries of a row
// (`bkc` = the row's bucket word of their first group, RC words apart).
template <int SEGW>
BIV_DEV void seg_bounds(const uint32_t (&r)[SEGW], const unsigned long long* bkc, int RC, const float* ntab,
                        float invT, float (&bound)[SEGW]) {
    unsigned long long bw[SEGW / 4];
#pragma unroll
    for (int i = 0; i < SEGW / 4; ++i) bw[i] = bkc[i * RC];
#pragma unroll
    for (int e = 0; e < SEGW; ++e) {
        const uint32_t b = static_cast<uint32_t>(bw[e >> 2] >> (16 * (e & 3))) & 0xffffu;
        bound[e] = __fadd_rn(__fmul_rn(__uint_as_float(r[e]), invT), ntab[b]);
    }
}

// The key whose order (key_order) is o, for o != 0 (numbers).
BIV_DEV float key_value(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// Largest of SEGW values (NaN only if all are NaN) and the lowest index
// holding it (-1 if none): a tree, then a mask of the equal entries.
template <int SEGW>
BIV_DEV float seg_max(const float (&v)[SEGW], int lim, int& idx) {
    float t[SEGW];
#pragma unroll
    for (int e = 0; e < SEGW; ++e) t[e] = e < lim ? v[e] : __int_as_float(0x7fc00000);
#pragma unroll
    for (int w = SEGW / 2; w > 0; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
    const float m = t[0];
    uint32_t mask = 0;
#pragma unroll
    for (int e = 0; e < SEGW; ++e) mask |= (e < lim && v[e] == m) ? (1u << e) : 0u;
    idx = mask ? __ffs(mask) - 1 : -1;
    return m;
}

template <int SEGW>
BIV_DEV void seg_load(uint32_t taddr, uint32_t (&r)[SEGW]);
template <>
BIV_DEV void seg_load<32>(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld32_sync(taddr, r); }
template <>
BIV_DEV void seg_load<16>(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16x2_sync(taddr, r); }

// Winner among tile columns [cb, ce) of one tile-row of logits held in TMEM
// (columns n0 + cb .. of a row, valid below N; cb and ce multiples of 32),
// exactly as the selection kernel
// defines it: key = fl(fl(x * invT) + g), largest key, lowest index among
// equal keys, a NaN never beats a number.  The row is walked in 32-column
// chunks; with SEGW = 32 one thread owns the row (M = 128 accumulators), with
// SEGW = 16 two threads share it (M = 64 accumulators: threads l and l + 16
// take columns [c, c + 16) and [c + 16, c + 32) of every chunk) and their
// winners are merged at the end.  Every entry has the bound
// fl(fl(x * invT) + T[bucket]) >= its key (fp32 rounding is monotone).  Pass 1
// finds a thread's entry with the largest bound (its exact key is the lower
// bound LB) and each chunk's largest bound; pass 2 revisits only chunks whose
// largest bound reaches LB (for LB's own chunk, the largest other bound) and
// evaluates the exact key only of entries whose bound does.  T = 0 takes the
// largest logit.  TMEM loads are warp-wide: a chunk is reloaded when any lane
// of the warp needs it.  `bkrow` is the row's buckets, `cm` the thread's
// chunk maxima (shared memory).
// Bounds of the 32 entries of one chunk (columns col0 .. col0 + 31, col0 a
// multiple of 32) from Philox words drawn here: the same buckets as
// tile_buckets stores, without the shared-memory copy (for tiles whose
// epilogue runs under the next tile's MMAs anyway).
BIV_DEV void fly_bounds(const uint32_t (&r)[32], uint32_t col0, uint32_t pos, uint32_t req, const SelectArgs& sel,
                        const float* ntab, float (&bound)[32]) {
    constexpr int sh = 32 - kBucketBits;
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) {
        const U4 w = philox4x32_10((col0 >> 2) + static_cast<uint32_t>(g4), pos, req, 0u, sel.seed_lo, sel.seed_hi);
        bound[4 * g4 + 0] = __fadd_rn(__fmul_rn(__uint_as_float(r[4 * g4 + 0]), sel.invT), ntab[w.x >> sh]);
        bound[4 * g4 + 1] = __fadd_rn(__fmul_rn(__uint_as_float(r[4 * g4 + 1]), sel.invT), ntab[w.y >> sh]);
        bound[4 * g4 + 2] = __fadd_rn(__fmul_rn(__uint_as_float(r[4 * g4 + 2]), sel.invT), ntab[w.z >> sh]);
        bound[4 * g4 + 3] = __fadd_rn(__fmul_rn(__uint_as_float(r[4 * g4 + 3]), sel.invT), ntab[w.w >> sh]);
    }
}

// FLY: the bucket words are drawn per chunk (fly_bounds) instead of read
// from the tile's bucket table `bkrow` (SEGW = 32 only).
template <int SEGW, bool FLY = false>
BIV_DEV unsigned long long tile_row_winner(uint32_t taddr, int cb, int ce, int n0, int N, bool live, uint32_t req,
                                           uint32_t pos, const SelectArgs& sel, const float* ntab,
                                           const unsigned long long* bkrow, int RC, float* cm, float* logits_row,
                                           unsigned long long floor_key = 0) {
    static_assert(!FLY || SEGW == 32, "per-chunk bucket words need whole 32-column chunks per thread");
    const int hoff = SEGW == 16 ? static_cast<int>(threadIdx.x & 16) : 0;
    float bx = -INFINITY;       // largest logit (T = 0) or largest bound (T > 0)
    float bxv = 0.0f;           // the logit of that entry
    float bm2 = -INFINITY;      // the largest other bound of that entry's chunk
    int bi = -1;
#pragma unroll 1
    for (int c = cb; c < ce; c += kChunk) {
        uint32_t r[SEGW];
        seg_load<SEGW>(taddr + static_cast<uint32_t>(c), r);
        if (!live) continue;
        const int col0 = n0 + c + hoff;
        const int lim = N - col0;               // entries of this segment below N
        float val[SEGW];
        if (sel.greedy) {
#pragma unroll
            for (int e = 0; e < SEGW; ++e) val[e] = __uint_as_float(r[e]);
        } else if constexpr (FLY) {
            fly_bounds(r, static_cast<uint32_t>(col0), pos, req, sel, ntab, val);
        } else {
            seg_bounds<SEGW>(r, bkrow + ((c + hoff) / 4) * RC, RC, ntab, sel.invT, val);
        }
        int e = -1;
        const float m = seg_max<SEGW>(val, lim, e);
        if (!sel.greedy) cm[c / kChunk] = m;
        if (e >= 0 && (m > bx || bi < 0)) {
            bx = m;
            bi = col0 + e;
            float xv = 0.0f;          // r[e] without a dynamic register index
#pragma unroll
            for (int j = 0; j < SEGW; ++j) xv = (j == e) ? __uint_as_float(r[j]) : xv;
            bxv = xv;
            if (!sel.greedy) {
#pragma unroll
                for (int j = 0; j < SEGW; ++j) val[j] = (j == e) ? __int_as_float(0x7fc00000) : val[j];
                int e2;
                bm2 = seg_max<SEGW>(val, lim, e2);
            }
        }
        if (logits_row) {
#pragma unroll
            for (int h = 0; h < SEGW / 8; ++h) {
                const int col = col0 + h * 8;
                if (col < N) {
                    const uint32_t* v = r + h * 8;
                    float4* dst = reinterpret_cast<float4*>(logits_row + col);
                    dst[0] = make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                                         __uint_as_float(v[3]));
                    dst[1] = make_float4(__uint_as_float(v[4]), __uint_as_float(v[5]), __uint_as_float(v[6]),
                                         __uint_as_float(v[7]));
                }
            }
        }
    }
    unsigned long long best = 0;
    float thr = 0.0f;
    const bool act = live && n0 + cb + hoff < N && bi >= 0 && !sel.greedy;
    if (live && n0 + cb + hoff < N) {
        if (bi < 0) {
            best = static_cast<unsigned long long>(~static_cast<uint32_t>(n0 + cb + hoff));   // all NaN: key order 0
        } else if (sel.greedy) {
            best = pack_key(bx, static_cast<uint32_t>(bi));
        } else {
            // LB: the exact key of the entry with the largest bound.
            const uint32_t v = static_cast<uint32_t>(bi);
            const U4 w = philox4x32_10(v >> 2, pos, req, 0u, sel.seed_lo, sel.seed_hi);
            thr = __fadd_rn(__fmul_rn(bxv, sel.invT), gumbel_from_word(pick_word(w, v & 3u)));
            best = pack_key(thr, v);
            // a larger real key of the row found elsewhere (floor_key, a numeric
            // key) raises the bar for pass 2; no entry below it can win
            if (floor_key > best && (floor_key >> 32) != 0ull) {
                best = floor_key;
                thr = key_value(static_cast<uint32_t>(floor_key >> 32));
            }
        }
    }
    if (!sel.greedy) {
#pragma unroll 1
        for (int c = cb; c < ce; c += kChunk) {
            const int col0 = n0 + c + hoff;
            const bool own = bi >= col0 && bi < col0 + SEGW;
            const bool need = act && (own ? bm2 : cm[c / kChunk]) >= thr;
            if (!__any_sync(0xffffffffu, need)) continue;
            uint32_t r[SEGW];
            seg_load<SEGW>(taddr + static_cast<uint32_t>(c), r);
            if (!need) continue;
            float bound[SEGW];
            if constexpr (FLY)
                fly_bounds(r, static_cast<uint32_t>(col0), pos, req, sel, ntab, bound);
            else
                seg_bounds<SEGW>(r, bkrow + ((c + hoff) / 4) * RC, RC, ntab, sel.invT, bound);
            const int lim = N - col0;
            uint32_t hit = 0;
#pragma unroll
            for (int e = 0; e < SEGW; ++e)
                if (e < lim && bound[e] >= thr && col0 + e != bi) hit |= 1u << e;
            while (hit) {
                const int e = __ffs(hit) - 1;
                hit &= hit - 1;
                const uint32_t v = static_cast<uint32_t>(col0 + e);
                float xv = 0.0f;          // r[e] without a dynamic register index
#pragma unroll
                for (int j = 0; j < SEGW; ++j) xv = (j == e) ? __uint_as_float(r[j]) : xv;
                const U4 w = philox4x32_10(v >> 2, pos, req, 0u, sel.seed_lo, sel.seed_hi);
                const float key = __fadd_rn(__fmul_rn(xv, sel.invT), gumbel_from_word(pick_word(w, v & 3u)));
                const unsigned long long pk = pack_key(key, v);
                if (pk > best) {
                    best = pk;
                    thr = key;
                }
            }
        }
    }
    if (SEGW == 16) {             // the two threads of the row: the larger packed key
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, 16);
        best = umax64(best, other);
    }
    return best;
}

// EPI: 0 = bf16 C, 1 = fp32 C, 2 = SwiGLU of gate/up-interleaved B (bf16
// activation [M, N/2]; see biv_gemm_swiglu), 3 = Gumbel-max selection of each
// tile-row (optional fp32 C; see biv_lm_head_gumbel), 4 = RoPE of q and k, k
// and v into the KV cache (see biv_gemm_qkv_rope).
// CG = 1: one CTA per tile of 128 rows.  CG = 2: a cluster of two CTAs per
// tile of 256 rows (cta_group::2 MMAs of M = 256): each CTA copies its own
// 128 rows of A and its half of the tile's BN rows of B into its own shared
// memory, both CTAs' copies complete on the even CTA's stage barrier, the
// even CTA's MMA thread issues the pair MMAs (the tensor core reads the B
// halves of both CTAs, so every weight byte enters one SM's shared memory
// once per pair) and each CTA's epilogue drains its own 128 rows from its own
// tensor memory.  Per output element the MMAs, their k order and the single
// fp32 accumulator are those of CG = 1.
template <int EPI, int CG>
__global__ void __launch_bounds__(64 + epi_threads<EPI>(), 1)
gemm_nosplitk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                     void* __restrict__ C, const GemmArgs g, const SelectArgs sel, const RopeArgs rp) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int A_BYTES = g.KS * g.a_rows * kRowBytes;     // A region of a stage
    const int STAGE = A_BYTES + g.KS * (g.BN / CG) * kRowBytes;
    const int S = g.stages;
    uint8_t* tiles = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * STAGE + (g.a_rows < kBM ? kTailSlack : 0));
    uint64_t* empty = full + kMaxStages;
    uint64_t* tfull = empty + kMaxStages;     // [2]
    uint64_t* tempty = tfull + 2;             // [2]
    uint64_t* drain = tempty + 2;             // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* ntab = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + kBarBytes);   // EPI 3 only
    float* t8 = ntab + kBuckets;                                                             // EPI 3 only
    float* cmax = t8 + 256;                                                   // EPI 3: [256][8]
    unsigned long long* s_best = reinterpret_cast<unsigned long long*>(cmax + 2 * kBM * kMaxChunks);  // [128]
    unsigned long long* bk = s_best + kBM;                                                   // EPI 3 only
    unsigned long long* s_run = bk;             // EPI 3, CG = 2: [128] each row's best over the CTA's tiles
    constexpr int NT = epi_threads<EPI>();
    constexpr int TM = kBM * CG;                  // rows of one output tile
    // CG = 2: the pair's rank (0 = the even CTA, which owns the stage and
    // accumulator-empty barriers and issues the MMAs) and its tiles.
    const int rank = CG == 2 ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit = CG == 2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int n_units = CG == 2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int M = g.M, N = g.N, BN = g.BN;
    const int BNL = BN / CG;                      // B rows this CTA copies per tile
    const int m_tiles = (M + TM - 1) / TM;
    const int n_tiles = column_tiles(g);
    const int n_work = m_tiles * n_tiles;
    const int KB = g.KB;
    const int KS = g.KS;
    const int n_stage_blocks = g.first1 ? 1 + (KB - 1 + KS - 1) / KS : (KB + KS - 1) / KS;   // stages per tile
    const uint32_t tx_bytes = static_cast<uint32_t>(STAGE);
    const uint32_t tx_bytes1 = static_cast<uint32_t>((g.a_rows + g.BN) * kRowBytes);     // a one-k-block stage

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], CG == 2 ? 2 : NT);   // CG = 2: one arrival per CTA's epilogue
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (g.first1) {
            prefetch_tensormap(&tmA1);
            prefetch_tensormap(&tmB1);
        }
    }
    if (warp == 1) {
        if constexpr (CG == 2) {
            tmem_alloc_pair(tmem_slot, g.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, g.tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    if constexpr (CG == 2)
        cluster_sync();       // both CTAs' barriers are initialised before either signals the other's
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t pol_a = policy_evict_last();    // activations: reused by every CTA
    const uint64_t pol_b = policy_evict_first();   // weights: streamed once
    // The weights are not an output of the previous kernel: the B boxes of the
    // first tile's first stages are requested before waiting for it (their A
    // boxes, the previous kernel's output, after).  Each such stage's barrier
    // expects both from the start.
    int b_early = 0;
    if (warp == 0 && lane == 0 && unit < n_work) {
        const int n_blk0 = unit / m_tiles;      // a unit's first tile is a full one (the tail follows whole waves)
        b_early = min(S, n_stage_blocks);
        for (int sb = 0; sb < b_early; ++sb) {
            uint8_t* sa = tiles + sb * STAGE;
            int kb0, nkb;
            stage_range(g, sb, kb0, nkb);
            if constexpr (CG == 2) {
                // the even CTA expects both CTAs' bytes of the stage
                if (rank == 0) mbar_arrive_expect_tx(&full[sb], 2 * tx_bytes);
                tma_load_3d_pair(sa + A_BYTES, &tmB, mapa_shared(&full[sb], 0), 0, n_blk0 * BN + rank * BNL, kb0,
                                 pol_b);
            } else if (g.first1 && sb == 0) {
                mbar_arrive_expect_tx(&full[sb], tx_bytes1);
                tma_load_3d(sa + A_BYTES, &tmB1, &full[sb], 0, n_blk0 * BN, 0, pol_b);
            } else if (g.three_d) {
                mbar_arrive_expect_tx(&full[sb], tx_bytes);
                tma_load_3d(sa + A_BYTES, &tmB, &full[sb], 0, n_blk0 * BN, kb0, pol_b);
            } else {
                mbar_arrive_expect_tx(&full[sb], tx_bytes);
                tma_load_2d(sa + A_BYTES, &tmB, &full[sb], sb * kBK, n_blk0 * BN, pol_b);
            }
        }
    }
    pdl_wait();       // inputs of the previous kernel are complete and visible from here on
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int t = unit; t < n_work && ok; t += n_units) {
                const TileAt ti = tile_at(g, t, m_tiles);
                const int m_blk = ti.m_blk;
                const int bnl_t = ti.bn / CG;
                const CUtensorMap* tmBt = ti.bn == BN ? &tmB : &tmB1;
                const uint32_t tx_t = static_cast<uint32_t>(A_BYTES + KS * bnl_t * kRowBytes);
                for (int sb = 0; sb < n_stage_blocks; ++sb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_gemm_err, true, CG == 2)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = tiles + stage * STAGE;
                    int kb0, nkb;
                    stage_range(g, sb, kb0, nkb);
                    const bool b_done = t == unit && sb < b_early;   // B requested early
                    if constexpr (CG == 2) {
                        const uint32_t fb = mapa_shared(&full[stage], 0);
                        if (!b_done && rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * tx_t);
                        tma_load_3d_pair(sa, &tmA, fb, 0, m_blk * TM + rank * kBM, kb0, pol_a);
                        if (!b_done) tma_load_3d_pair(sa + A_BYTES, tmBt, fb, 0, ti.col0 + rank * bnl_t, kb0, pol_b);
                    } else if (g.first1 && sb == 0) {
                        if (!b_done) mbar_arrive_expect_tx(&full[stage], tx_bytes1);
                        tma_load_3d(sa, &tmA1, &full[stage], 0, m_blk * kBM, 0, pol_a);
                        if (!b_done) tma_load_3d(sa + A_BYTES, &tmB1, &full[stage], 0, ti.col0, 0, pol_b);
                    } else if (g.three_d) {
                        if (!b_done) mbar_arrive_expect_tx(&full[stage], tx_bytes);
                        tma_load_3d(sa, &tmA, &full[stage], 0, m_blk * kBM, kb0, pol_a);
                        if (!b_done) tma_load_3d(sa + A_BYTES, &tmB, &full[stage], 0, ti.col0, kb0, pol_b);
                    } else {
                        if (!b_done) mbar_arrive_expect_tx(&full[stage], tx_bytes);
                        tma_load_2d(sa, &tmA, &full[stage], sb * kBK, m_blk * kBM, pol_a);
                        if (!b_done) tma_load_2d(sa + A_BYTES, &tmB, &full[stage], sb * kBK, ti.col0, pol_b);
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
                if (CG == 1 || rank == 0) {
                    long long first = issued > S ? issued - S : 0;
                    for (long long i = first; i < issued; ++i)
                        mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1));
                } else {
                    // the odd CTA's copies complete on the even CTA's barriers:
                    // give them time to land
                    const uint64_t t0 = globaltimer();
                    while (globaltimer() - t0 < 50000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- MMA issuer
        // The whole warp walks the loop with warp-uniform operands: every lane
        // observes each barrier (a time-out anywhere stops all of them) and
        // one elected lane issues the MMAs and their commits.  With CG = 2 the
        // even CTA's warp issues the pair's MMAs and signals both CTAs.
        if (CG == 1 || rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int t = unit; t < n_work && ok; t += n_units) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, &g_gemm_err, true, CG == 2))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const TileAt ti = tile_at(g, t, m_tiles);
                const uint32_t idesc_t = ti.bn == BN ? g.idesc : g.idesc_tail;
                const int bnl_t = ti.bn / CG;
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int sb = 0; sb < n_stage_blocks; ++sb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&full[stage], phase, abort_flag, &g_gemm_err, true, CG == 2))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(tiles + stage * STAGE);
                    const uint32_t b_addr = a_addr + static_cast<uint32_t>(A_BYTES);
                    int kb0, nkb;
                    stage_range(g, sb, kb0, nkb);
                    for (int j = 0; j < nkb; ++j) {
                        const int kb = kb0 + j;
                        const uint64_t a_desc = sw128_kmajor_desc(a_addr + static_cast<uint32_t>(j * g.a_rows * kRowBytes));
                        const uint64_t b_desc = sw128_kmajor_desc(b_addr + static_cast<uint32_t>(j * bnl_t * kRowBytes));
#pragma unroll
                        for (int k = 0; k < kBK / 16; ++k) {
                            // +32 bytes along K inside the swizzle row = +2 in 16-byte units.
                            if constexpr (CG == 2)
                                umma_bf16_pair_elect(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc_t,
                                                     (kb > 0 || k > 0) ? 1u : 0u);
                            else
                                umma_bf16_elect(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc_t,
                                                (kb > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    any = true;
                    if constexpr (CG == 2) {
                        // the stage is free in both CTAs once these MMAs are done
                        umma_commit_pair_elect(mapa_shared(&empty[stage], 0));
                        umma_commit_pair_elect(mapa_shared(&empty[stage], 1));
                    } else {
                        umma_commit_elect(&empty[stage]);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (CG == 2) {
                    umma_commit_pair_elect(mapa_shared(&tfull[acc], 0));
                    umma_commit_pair_elect(mapa_shared(&tfull[acc], 1));
                } else {
                    umma_commit_elect(&tfull[acc]);
                }
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                // all MMAs issued so far have finished
                if constexpr (CG == 2)
                    umma_commit_pair_elect(mapa_shared(drain, 0));
                else
                    umma_commit_elect(drain);
                if (lane == 0) mbar_wait_drain(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        if constexpr (EPI == 3) {
            // Largest noise of each bucket, while the first tile's data arrives.
            if (!sel.greedy) fill_noise_table<NT>(ntab, t8);
        }
        const float* inv_freq = nullptr;
        if constexpr (EPI == 4) {
            // RoPE frequencies of the pairs; the first tile's vote publishes them.
            __shared__ float s_inv_freq[128];                  // head_dim <= 256
            for (int i = static_cast<int>(threadIdx.x) - 64; i < rp.hd / 2; i += NT)
                s_inv_freq[i] = rope_inv_freq(i, rp.hd, rp.theta);
            inv_freq = s_inv_freq;
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        unsigned long long run = 0;                 // EPI 3, CG = 2: see below
        int run_mblk = -1;
        for (int t = unit; t < n_work; t += n_units) {
            const TileAt ti = tile_at(g, t, m_tiles);
            const int m_blk = ti.m_blk;
            const int bnt = ti.bn, col0 = ti.col0;                 // this tile's width and first column
            const int row_base = m_blk * TM + rank * kBM;          // first row of this CTA's 128
            if constexpr (EPI == 3 && CG == 1) {
                // This tile's noise buckets while its MMAs run; the vote below is
                // also the barrier that makes them (and the table) visible.
                // (CG = 2 draws them per chunk: the epilogue of a tile runs
                // under the next tile's MMAs.)
                if (!sel.greedy)
                    tile_buckets<NT>(bk, g.a_rows, min(kBM, M - m_blk * kBM), bnt, col0, N, m_blk * kBM, sel);
            }
            // One thread polls the accumulator barrier; the vote hands its
            // outcome to the other epilogue threads (no polling traffic beside
            // the copies).
            bool ok = threadIdx.x == 64 ? mbar_wait(&tfull[acc], acc_phase, abort_flag, &g_gemm_err, false, CG == 2)
                                        : true;
            ok = epilogue_all<NT>(ok);
            if (!ok) break;
            tc_fence_after();
            // M = 128 MMAs put tile row r in TMEM lane r; M = 64 MMAs put row r in
            // lane 32 (r / 16) + r % 16, so each warp owns 16 rows in lanes 0..15.
            const int rloc = g.m64 ? q * 16 + lane : q * 32 + lane;
            const int row = row_base + rloc;
            const bool live = row < M && (!g.m64 || lane < 16);
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
            if constexpr (EPI == 3) {
                // with M = 64 accumulators the two half-warps share each row
                const int srloc = g.m64 ? q * 16 + (lane & 15) : rloc;
                const int srow = row_base + srloc;
                const bool slive = srow < M;
                const uint32_t req = slive ? sel.row_req[srow] : 0u;
                const uint32_t pos = slive ? static_cast<uint32_t>(sel.row_pos[srow]) + 1u : 0u;
                float* lrow = (C != nullptr && slive) ? static_cast<float*>(C) + static_cast<long long>(srow) * N
                                                      : nullptr;
                // warps 2-5 take the tile's first half of 32-column chunks, warps
                // 6-9 the rest; their winners meet in shared memory
                const int eset = (warp - 2) >> 2;
                const int nch = bnt / kChunk, h1 = (nch + 1) / 2;
                const int cb = eset ? h1 * kChunk : 0, ce = eset ? bnt : h1 * kChunk;
                float* cmt = cmax + (eset * kBM + q * 32 + lane) * kMaxChunks;
                unsigned long long best;
                if constexpr (CG == 2) {
                    // A CTA pair keeps its row tile from one tile to the next as long
                    // as the pairs divide the row tiles: the row's best key over the
                    // CTA's earlier tiles (a real key of the row) then bounds pass 2
                    // from below, so fewer chunks are revisited.
                    if (run_mblk != m_blk) run = 0;
                    else if (live) run = umax64(run, s_run[rloc]);
                    run_mblk = m_blk;
                    best = tile_row_winner<32, true>(taddr, cb, ce, col0, N, slive, req, pos, sel, ntab,
                                                     nullptr, 0, cmt, lrow, run);
                }
                else
                    best = g.m64 ? tile_row_winner<16>(taddr, cb, ce, col0, N, slive, req, pos, sel, ntab,
                                                       bk + srloc, g.a_rows, cmt, lrow)
                                 : tile_row_winner<32>(taddr, cb, ce, col0, N, slive, req, pos, sel, ntab,
                                                       bk + srloc, g.a_rows, cmt, lrow);
                if (eset == 1 && live) s_best[rloc] = best;
                epilogue_bar<NT>();   // both halves' winners are in; every row is done with the buckets
                if (eset == 0 && live) {
                    const unsigned long long w = umax64(best, s_best[rloc]);
                    sel.cand[static_cast<long long>(srow) * n_tiles + ti.slot] = w;
                    if constexpr (CG == 2) s_run[rloc] = w;    // read by both halves at the next tile
                }
            } else if constexpr (EPI == 4) {
                // With M = 64 accumulators the two half-warps share each row:
                // threads 16..31 take pairs 4..7 of every 16-column group.
                const int prow = g.m64 ? row_base + q * 16 + (lane & 15) : row;
                const bool plive = prow < M;
                const int jb = g.m64 ? 4 * (lane >> 4) : 0;
                int slot = 0, pos = 0;
                bool write_kv = false;
                if (plive) {
                    pos = rp.row_pos[prow];
                    slot = rp.row_slot[prow];
                    const bool keep = !rp.rows_keep || (prow % rp.K) < rp.rows_keep[prow / rp.K];
                    const bool cache_ok = slot >= 0 && slot < rp.n_slots && pos >= 0 && pos < rp.max_len;
                    if (keep && !cache_ok && jb == 0) atomicOr(&g_gemm_err, BIV_DEVERR_INDEX);
                    write_kv = keep && cache_ok;
                }
                int cb4, ce4;
                eset_columns(bnt, 16, (warp - 2) >> 2, cb4, ce4);
                if (g.m64) {
                    RopeAngles<4> ang;
#pragma unroll 1
                    for (int c = cb4; c < ce4; c += 16) {
                        const int col = col0 + c;
                        uint32_t ra[4], rb[4];
                        tmem_ld16x2_x4_pair_sync(taddr + static_cast<uint32_t>(c),
                                                 taddr + static_cast<uint32_t>(c + 8), ra, rb);
                        if (plive && col < N)
                            qkv_group<4>(ra, rb, jb, col, prow, slot, pos, write_kv, rp, inv_freq, ang);
                    }
                } else {
                    RopeAngles<8> ang;
#pragma unroll 1
                    for (int c = cb4; c < ce4; c += 16) {
                        const int col = col0 + c;
                        uint32_t r[16];
                        tmem_ld16(taddr + static_cast<uint32_t>(c), r);
                        tmem_ld_wait();
                        if (live && col < N)
                            qkv_group<8>(r, r + 8, 0, col, row, slot, pos, write_kv, rp, inv_freq, ang);
                    }
                }
            } else if constexpr (EPI == 2) {
                // Columns [32j, 32j + 16) of the tile are gate rows, [32j + 16, 32j + 32)
                // the matching up rows: act = bf16(silu(bf16(g)) * bf16(u)).
                const int F = N / 2;
                int cb2, ce2;
                eset_columns(bnt, 32, (warp - 2) >> 2, cb2, ce2);
                if (g.m64) {
                    // the two half-warps share each row: threads 16..31 take
                    // gate columns 8..15 of every 32-column group and their up columns
                    const int prow = row_base + q * 16 + (lane & 15);
                    const int hi = lane >> 4;
#pragma unroll 1
                    for (int c = cb2; c < ce2; c += 32) {
                        uint32_t gr[8], ur[8];
                        tmem_ld16x2_x8_pair_sync(taddr + static_cast<uint32_t>(c),
                                                 taddr + static_cast<uint32_t>(c + 16), gr, ur);
                        const int col = col0 + c;
                        if (prow < M && col < N) {
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                o[e] = swiglu_pack(
                                    pack_bf16x2(__uint_as_float(gr[2 * e]), __uint_as_float(gr[2 * e + 1])),
                                    pack_bf16x2(__uint_as_float(ur[2 * e]), __uint_as_float(ur[2 * e + 1])));
                            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(C) + static_cast<long long>(prow) * F +
                                                      col / 2 + 8 * hi) = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                } else
#pragma unroll 1
                for (int c = cb2; c < ce2; c += 32) {
                    uint32_t gr[16], ur[16];
                    tmem_ld16(taddr + static_cast<uint32_t>(c), gr);
                    tmem_ld16(taddr + static_cast<uint32_t>(c + 16), ur);
                    tmem_ld_wait();
                    const int col = col0 + c;
                    if (live && col < N) {
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
            int cb0, ce0;
            eset_columns(bnt, 16, (warp - 2) >> 2, cb0, ce0);
#pragma unroll 1
            for (int c = cb0; c < ce0; c += 16) {
                uint32_t r[16];
                tmem_ld16(taddr + static_cast<uint32_t>(c), r);
                tmem_ld_wait();
                if (live) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int col = col0 + c + h * 8;
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
            if constexpr (CG == 2) {
                // every epilogue thread of this CTA is done with the accumulator:
                // one arrival on the even CTA's barrier
                epilogue_bar<NT>();
                if (threadIdx.x == 64) mbar_arrive_cluster(mapa_shared(&tempty[acc], 0));
            } else {
                mbar_arrive(&tempty[acc]);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    if constexpr (CG == 2) {
        // neither CTA leaves while the other may still read its shared memory
        // (pair MMAs) or signal its barriers
        cluster_sync();
        tc_fence_after();
        if (warp == 1) tmem_dealloc_pair(tmem_base, g.tmem_cols);
    } else {
        __syncthreads();
        tc_fence_after();
        if (warp == 1) tmem_dealloc(tmem_base, g.tmem_cols);
    }
}

// --------------------------------------------------------------- host side
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

// Problems of more than one 128-row tile (with K a multiple of 64) run as CTA
// pairs: 256-row tiles, each weight tile copied once per pair.
inline bool use_pair(int M, int K) { return M > kBM && K % kBK == 0; }

// Once per device and kernel instance (from any host thread): the kernel's
// opt-in shared memory size and, for pair kernels, how many 2-CTA clusters of
// it can be resident at once (the persistent grid's size).  Returns a
// biv_status.
template <int EPI, int CG>
int kernel_setup(int dev, int smem_max, int* resident_units) {
    static std::mutex mu;
    static int units[kMaxDevices] = {};           // 0 = not yet configured
    if (dev < 0 || dev >= kMaxDevices) return BIV_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(mu);
    if (units[dev] == 0) {
        auto kern = gemm_nosplitk_kernel<EPI, CG>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
        if (e != cudaSuccess) return cuda_status(e);
        int n = num_sms();
        if (CG == 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(2 * num_sms()));
            cfg.blockDim = dim3(64 + epi_threads<EPI>());
            cfg.dynamicSmemBytes = static_cast<size_t>(smem_max);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess) return cuda_status(e);
            if (n <= 0) return BIV_ERR_DEVICE;
        }
        units[dev] = n;
    }
    *resident_units = units[dev];
    return BIV_OK;
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// The narrow tail of the fused selection's CTA-pair schedule.  With work
// tiles on a wave of kPairWave pairs, the last wave holds r = work mod wave
// tiles; when those are whole column tiles (row tiles fastest) they are re-cut
// into the narrowest tiles (a multiple of 32 columns, at least 64) of which
// one wave still holds all, so that every pair ends with one short tile
// instead of some pairs with a whole one.  W = 1024 (2004 tiles of 256 columns
// on 76 pairs, 28 in the last wave): 76 tiles of 96 columns; W = 256 (501 on
// 76, 45 in the last wave): 72 of 160.  Each element's arithmetic does not
// depend on the tile width.
struct TailPlan {
    int nt_full, bn_tail, n_cols;     // full column tiles, tail width (0: none), column tiles in all
};

inline TailPlan tail_plan(int M, int N, int BN, bool pairs) {
    const int n_tiles = static_cast<int>(ceil_div(N, BN));
    TailPlan p{n_tiles, 0, n_tiles};
    if (!pairs) return p;
    const long long m_tiles = ceil_div(M, 2 * kBM);
    const long long work = m_tiles * n_tiles;
    const long long wave = std::min<long long>(work, kPairWave);
    const long long r = work % wave;
    if (r == 0 || r % m_tiles != 0) return p;
    const int nt_full = n_tiles - static_cast<int>(r / m_tiles);
    const long long tail_cols = N - static_cast<long long>(nt_full) * BN;
    for (int bt = 64; bt < BN; bt += 32) {
        const long long nt_tail = ceil_div(tail_cols, bt);
        if (m_tiles * nt_tail <= wave) return TailPlan{nt_full, bt, nt_full + static_cast<int>(nt_tail)};
    }
    return p;
}

template <int EPI, int CG>
int launch_gemm_cg(const void* A, const void* B, void* C, int M, int N, int K, int BN, cudaStream_t stream,
                   const SelectArgs& sel, const RopeArgs& rp, int* n_cols) {
    GemmArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.BN = BN;
    g.a_rows = (CG == 2 || M >= kBM) ? kBM : ((M + 7) / 8) * 8;
    g.KB = (K + kBK - 1) / kBK;
    g.three_d = (K % kBK == 0) ? 1 : 0;
    const int BNL = BN / CG;                        // B rows one CTA copies per tile
    // The TMA unit spends a fixed ~275 ns per box whatever its size, so a box
    // should be as large as possible.  With one row tile (M <= 128, weight
    // streaming) each stage takes as many k-blocks as let two stages fit the
    // ring; the MMA may then read past the packed A rows of the last stage, so
    // the ring keeps a tail.  Otherwise (full 128-row tiles) one or two
    // k-blocks per stage and as many stages as fit.
    int ks = 1;
    const int tail = g.a_rows < kBM ? kTailSlack : 0;
    // EPI 3 keeps the noise table, chunk maxima and (CG = 1) one tile of noise
    // buckets beside the ring, and takes all of the opt-in shared memory.
    const int extra = EPI == 3 ? kNoiseTableBytes + 2 * kBM * kMaxChunks * 4 + kBM * 8 +
                                     (CG == 1 ? g.a_rows * BN * 2 : kBM * 8)
                               : 0;
    // The ring takes the opt-in shared memory left after the 1 KiB alignment
    // pad, the barriers and (non-selection epilogues) up to 1 KiB of the
    // kernel's static shared memory.
    const int ring = EPI == 3 ? kMaxSmem - 1024 - kBarBytes - extra : kMaxSmem - 2048 - kBarBytes;
    const long long work = static_cast<long long>((M + kBM * CG - 1) / (kBM * CG)) * ((N + BN - 1) / BN);   // full-width tiles
    const int smem_max = EPI == 3 ? kMaxSmem : kMaxSmem - 1024;
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_status(de);
    int units = 0;
    const int st = kernel_setup<EPI, CG>(dev, smem_max, &units);
    if (st != BIV_OK) return st;
    if (CG == 2) {
        // Pairs: two k-blocks per box while the ring holds three stages.
        if (ring / (2 * (g.a_rows + BNL) * kRowBytes) >= 3) ks = 2;
    } else if (g.three_d && M <= kBM) {        // one row tile: weight streaming
        const int per_kb = (g.a_rows + BN) * kRowBytes;
        ks = std::max(1, (ring - tail) / (2 * per_kb));
        ks = std::min(ks, std::min(g.KB, 256));
    } else if (g.three_d && work <= num_sms() && ring / (2 * (g.a_rows + BN) * kRowBytes) >= 3) {
        // Several row tiles in a single wave: two k-blocks per box halve the
        // boxes while the ring still holds three stages (measured 20-30 %
        // faster at M = 256-512 on 4096-wide weights); with several tiles per
        // CTA, or fewer stages, one-k-block stages keep the copies further ahead.
        ks = 2;
    }
    g.KS = ks;
    // A one-k-block first stage pays off where the MMA chain, not the copy,
    // sets the pace (narrow tiles with many k-blocks per stage).
    g.first1 = (CG == 1 && g.three_d && ks >= 4 && g.KB > 1) ? 1 : 0;
    g.m64 = g.a_rows <= 64 ? 1 : 0;
    g.stages = std::min(kMaxStages, std::max(1, (ring - tail) / stage_bytes(ks, g.a_rows, BNL)));
    g.idesc = idesc_bf16_f32(CG == 2 ? 2 * kBM : (g.m64 ? 64 : kBM), BN);
    g.tmem_cols = tmem_cols_for(BN);
    // the narrow tail: the fused selection on pairs, when the wave it is
    // planned for is the resident one (a unit's first tile is then a full one)
    const TailPlan tp = tail_plan(M, N, BN, EPI == 3 && CG == 2 && units == kPairWave);
    g.nt_full = tp.nt_full;
    g.bn_tail = tp.bn_tail;
    g.idesc_tail = tp.bn_tail ? idesc_bf16_f32(2 * kBM, tp.bn_tail) : g.idesc;
    if (n_cols) *n_cols = tp.n_cols;
    CUtensorMap ta, tb, ta1, tb1;
    if (!encode_kmajor(&ta, A, K, M, g.a_rows, ks, g.three_d) || !encode_kmajor(&tb, B, K, N, BNL, ks, g.three_d)) {
        set_cuda_error(cudaErrorInvalidValue);
        return BIV_ERR_CUDA;
    }
    ta1 = ta;
    tb1 = tb;
    if (g.first1 &&
        (!encode_kmajor(&ta1, A, K, M, g.a_rows, 1, true) || !encode_kmajor(&tb1, B, K, N, BN, 1, true))) {
        set_cuda_error(cudaErrorInvalidValue);
        return BIV_ERR_CUDA;
    }
    // the tail's B boxes (first1 is never set with pairs)
    if (g.bn_tail && !encode_kmajor(&tb1, B, K, N, g.bn_tail / CG, ks, g.three_d)) {
        set_cuda_error(cudaErrorInvalidValue);
        return BIV_ERR_CUDA;
    }
    const int smem = 1024 + g.stages * stage_bytes(ks, g.a_rows, BNL) + tail + kBarBytes + extra;
    auto kern = gemm_nosplitk_kernel<EPI, CG>;
    const dim3 block(64 + epi_threads<EPI>());
    if (CG == 2) {
        const int grid = 2 * static_cast<int>(std::min<long long>(work, units));
        return launch_cluster_pdl(kern, dim3(grid), block, static_cast<size_t>(smem), stream, 2, ta, tb, ta1, tb1, C,
                                  g, sel, rp);
    }
    const int grid = static_cast<int>(std::min<long long>(work, num_sms()));
    return launch_pdl(kern, dim3(grid), block, static_cast<size_t>(smem), stream, ta, tb, ta1, tb1, C, g, sel, rp);
}

// Pair tile widths: multiples of 32 in [64, 256] (each CTA copies BN / 2 rows
// of B, whole 16-row groups).  Other widths run one CTA per 128-row tile.
inline bool pair_bn_ok(int BN) { return BN % 32 == 0 && BN >= 64 && BN <= 256; }

template <int EPI>
int launch_gemm(const void* A, const void* B, void* C, int M, int N, int K, int BN, cudaStream_t stream,
                const SelectArgs& sel = SelectArgs{}, const RopeArgs& rp = RopeArgs{}, int* n_cols = nullptr) {
    if (use_pair(M, K) && pair_bn_ok(BN))
        return launch_gemm_cg<EPI, 2>(A, B, C, M, N, K, BN, stream, sel, rp, n_cols);
    return launch_gemm_cg<EPI, 1>(A, B, C, M, N, K, BN, stream, sel, rp, n_cols);
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

// Packed row p of the QKV weight: the q and k part is [gq][head][16], head h
// (q heads, then k heads) and frequency group gq: rows e = 0..7 are the head's
// dims 8 gq + e, rows e = 8..15 its dims hd/2 + 8 gq + e - 8 (the RoPE
// partners); the v heads are unchanged.
__global__ void rope_pack_kernel(const __nv_bfloat16* __restrict__ src, __nv_bfloat16* __restrict__ dst, int Hq,
                                 int Hkv, int hd, int K) {
    pdl_wait();
    const long long p = blockIdx.x;
    long long s = p;
    if (p < static_cast<long long>(Hq + Hkv) * hd) {
        const int nqk = Hq + Hkv;
        const int gi = static_cast<int>(p / 16), e = static_cast<int>(p % 16);
        const int gq = gi / nqk, h = gi - gq * nqk;
        const int dim = e < 8 ? 8 * gq + e : hd / 2 + 8 * gq + (e - 8);
        s = static_cast<long long>(h) * hd + dim;
    }
    const uint4* in = reinterpret_cast<const uint4*>(src + s * K);
    uint4* out = reinterpret_cast<uint4*>(dst + p * K);
    for (int c = threadIdx.x; c < K / 8; c += blockDim.x) out[c] = in[c];
}

// Largest of the row's n_tiles packed tile winners, taken by one warp: eight
// independent loads in flight per lane, then the warp maximum (a maximum is
// exact in any order).
BIV_DEV unsigned long long row_winner(const unsigned long long* __restrict__ row_cand, int n_tiles, int lane) {
    unsigned long long b[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int t = lane;
    for (; t + 7 * 32 < n_tiles; t += 8 * 32) {
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = umax64(b[j], row_cand[t + 32 * j]);
    }
    for (; t < n_tiles; t += 32) b[0] = umax64(b[0], row_cand[t]);
#pragma unroll
    for (int j = 1; j < 8; ++j) b[0] = umax64(b[0], b[j]);
    return warp_max64(b[0]);
}

// tokens[row] = the index of the largest of the row's tile winners (0 for a
// row with no number); one warp per row.
__global__ void tile_winners_kernel(const unsigned long long* __restrict__ cand, int M, int n_tiles,
                                    int32_t* __restrict__ tokens) {
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x * (blockDim.x / 32) + static_cast<int>(threadIdx.x / 32);
    const int lane = threadIdx.x & 31;
    if (row >= M) return;
    const unsigned long long b = row_winner(cand + static_cast<long long>(row) * n_tiles, n_tiles, lane);
    if (lane == 0) tokens[row] = b ? static_cast<int32_t>(~static_cast<uint32_t>(b & 0xffffffffull)) : 0;
}

constexpr int kMaxAcceptRows = 8192;              // K of one request in the fused winners + accept kernel

// One CTA per request: its warps take the per-row winners of the request's K
// rows (as tile_winners_kernel, one warp per row), then one thread takes the
// coupled accept (as verify_accept_kernel): accept length L = first j with
// target != draft, + 1, else K; new length p0 + L.  Same integer results as
// the two kernels.  Dynamic shared memory: K tokens.
__global__ void __launch_bounds__(1024)
winners_accept_kernel(const unsigned long long* __restrict__ cand, int n_tiles, int32_t* __restrict__ tokens,
                      const int32_t* __restrict__ draft, const int32_t* __restrict__ p0, int K,
                      int32_t* __restrict__ accept_len, int32_t* __restrict__ new_len) {
    extern __shared__ int32_t s_tok[];
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < K; j += blockDim.x / 32) {
        const long long row = static_cast<long long>(r) * K + j;
        const unsigned long long b = row_winner(cand + row * n_tiles, n_tiles, lane);
        if (lane == 0) {
            const int32_t tok = b ? static_cast<int32_t>(~static_cast<uint32_t>(b & 0xffffffffull)) : 0;
            tokens[row] = tok;
            s_tok[j] = tok;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int L = K;
        for (int j = 0; j < K; ++j) {
            if (s_tok[j] != draft[static_cast<long long>(r) * K + j]) {
                L = j + 1;
                break;
            }
        }
        accept_len[r] = L;
        new_len[r] = p0[r] + L;
    }
}

}  // namespace
}  // namespace biv

using namespace biv;

extern "C" int biv_gemm_tile_n(int M, int N, int K) {
    BIV_TRACE_CALL();
    const long long m_tiles = std::max<long long>(1, ceil_div(M, kBM));
    if (m_tiles == 1) {
        // Weight streaming: one wave of tiles, each as wide as that allows.
        const int bn = static_cast<int>(std::min<long long>(256, std::max<long long>(16, ceil_div(ceil_div(N, kWave), 16) * 16)));
        if (ceil_div(N, bn) <= kWave) return bn;
    }
    if (use_pair(M, K)) {
        // CTA pairs (256-row tiles): the width in [64, 256], a multiple of 32,
        // that best fills whole waves of 76 pairs (mildly preferring wide tiles).
        const long long m_pairs = ceil_div(M, 2 * kBM);
        int best = 256;
        double best_score = -1.0;
        for (int bn = 256; bn >= 64; bn -= 32) {
            const long long tiles = m_pairs * ceil_div(N, bn);
            const long long waves = ceil_div(tiles, kPairWave);
            const double fill = static_cast<double>(tiles) / static_cast<double>(waves * kPairWave);
            const double score = fill * bn / (bn + 32.0);
            if (score > best_score + 1e-9) {
                best_score = score;
                best = bn;
            }
        }
        return best;
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
    BIV_TRACE_CALL();
    int st = check_gemm(A, B, C, out_dtype, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    if (bn < 16 || bn > 256 || bn % 16 != 0) return BIV_ERR_VALUE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return out_dtype == BIV_F32 ? launch_gemm<1>(A, B, C, M, N, K, bn, s)
                                : launch_gemm<0>(A, B, C, M, N, K, bn, s);
}

extern "C" int biv_gemm_nosplitk(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K,
                                 biv_stream_t stream) {
    BIV_TRACE_CALL();
    int st = check_gemm(A, B, C, out_dtype, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    return biv_gemm_nosplitk_bn(A, B, C, out_dtype, M, N, K, biv_gemm_tile_n(M, N, K), stream);
}

extern "C" int biv_swiglu_pack_weights(const void* w_gu, void* w_packed, int F, int K, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (F <= 0 || K <= 0 || F % 16 != 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (!w_gu || !w_packed) return BIV_ERR_NULL;
    if (!aligned16(w_gu) || !aligned16(w_packed)) return BIV_ERR_ALIGN;
    if (w_gu == w_packed) return BIV_ERR_VALUE;
    return launch_pdl(swiglu_pack_kernel, dim3(2 * F), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                      static_cast<const __nv_bfloat16*>(w_gu), static_cast<__nv_bfloat16*>(w_packed), F, K);
}

extern "C" int biv_gemm_swiglu(const void* A, const void* B_packed, void* act, int M, int F, int K,
                               biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (F <= 0 || F % 16 != 0) return BIV_ERR_SHAPE;
    const int N = 2 * F;
    int st = check_gemm(A, B_packed, act, BIV_BF16, M, N, K);
    if (st != BIV_OK || M == 0) return st;
    const int bn = static_cast<int>(std::min<long long>(256, ceil_div(biv_gemm_tile_n(M, N, K), 32) * 32));
    return launch_gemm<2>(A, B_packed, act, M, N, K, bn, reinterpret_cast<cudaStream_t>(stream));
}

// Tile width of the fused LM head: the GEMM's rounded up to a multiple of 32
// (whole TMEM loads); with one CTA per full 128-row tile at most 128 (the
// buckets of one tile stay within 32 KiB of shared memory; CTA pairs draw
// them per chunk instead).
static int lm_head_tile_n(int M, int N, int K) {
    const int bn = static_cast<int>(std::min<long long>(256, ceil_div(biv_gemm_tile_n(M, N, K), 32) * 32));
    if (use_pair(M, K) && pair_bn_ok(bn)) return bn;
    return M >= 128 ? std::min(bn, 128) : bn;
}

extern "C" size_t biv_lm_head_gumbel_workspace_size(int M, int N, int K) {
    if (M <= 0 || N <= 0 || K <= 0) return 0;
    // one winner slot per column tile, with the narrow tail where it is planned
    const int bn = lm_head_tile_n(M, N, K);
    const long long n_cols = tail_plan(M, N, bn, use_pair(M, K) && pair_bn_ok(bn)).n_cols;
    return static_cast<size_t>(M) * static_cast<size_t>(n_cols) * sizeof(unsigned long long);
}

extern "C" int biv_lm_head_gumbel(const void* A, const void* B, float* logits, int M, int N, int K,
                                  const uint32_t* row_req, const int32_t* row_pos, uint64_t seed, float temperature,
                                  int32_t* tokens, void* workspace, size_t ws_bytes, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (M < 0 || N <= 0 || K <= 0 || N % 8 != 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (!(temperature >= 0.0f) || !(temperature < INFINITY)) return BIV_ERR_VALUE;
    if (M == 0) return BIV_OK;
    if (!A || !B || !row_req || !row_pos || !tokens || !workspace) return BIV_ERR_NULL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(workspace) || (logits && !aligned16(logits)))
        return BIV_ERR_ALIGN;
    if (ws_bytes < biv_lm_head_gumbel_workspace_size(M, N, K)) return BIV_ERR_SHAPE;
    const int bn = lm_head_tile_n(M, N, K);
    int n_tiles = static_cast<int>(ceil_div(N, bn));     // column tiles (winner slots per row) of the launch
    SelectArgs sel;
    sel.row_req = row_req;
    sel.row_pos = row_pos;
    sel.cand = static_cast<unsigned long long*>(workspace);
    sel.seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
    sel.seed_hi = static_cast<uint32_t>(seed >> 32);
    sel.greedy = temperature == 0.0f;
    sel.invT = sel.greedy ? 0.0f : 1.0f / temperature;    // fl(1/T), IEEE division on the host
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int st = launch_gemm<3>(A, B, logits, M, N, K, bn, s, sel, RopeArgs{}, &n_tiles);
    if (st != BIV_OK) return st;
    return launch_pdl(tile_winners_kernel, dim3((M + 7) / 8), dim3(256), 0, s,
                      static_cast<const unsigned long long*>(workspace), M, n_tiles, tokens);
}

extern "C" int biv_lm_head_gumbel_accept(const void* A, const void* B, float* logits, int M, int N, int K,
                                         const uint32_t* row_req, const int32_t* row_pos, uint64_t seed,
                                         float temperature, int32_t* tokens, const int32_t* draft, const int32_t* p0,
                                         int n_req, int rows_per_req, int32_t* accept_len, int32_t* new_len,
                                         void* workspace, size_t ws_bytes, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (M < 0 || N <= 0 || K <= 0 || N % 8 != 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (n_req < 0 || rows_per_req < 1 || static_cast<long long>(n_req) * rows_per_req != M) return BIV_ERR_SHAPE;
    if (!(temperature >= 0.0f) || !(temperature < INFINITY)) return BIV_ERR_VALUE;
    if (M == 0) return BIV_OK;
    if (!A || !B || !row_req || !row_pos || !tokens || !workspace || !draft || !p0 || !accept_len || !new_len)
        return BIV_ERR_NULL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(workspace) || (logits && !aligned16(logits)))
        return BIV_ERR_ALIGN;
    if (ws_bytes < biv_lm_head_gumbel_workspace_size(M, N, K)) return BIV_ERR_SHAPE;
    const int bn = lm_head_tile_n(M, N, K);
    int n_tiles = static_cast<int>(ceil_div(N, bn));     // column tiles (winner slots per row) of the launch
    SelectArgs sel;
    sel.row_req = row_req;
    sel.row_pos = row_pos;
    sel.cand = static_cast<unsigned long long*>(workspace);
    sel.seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
    sel.seed_hi = static_cast<uint32_t>(seed >> 32);
    sel.greedy = temperature == 0.0f;
    sel.invT = sel.greedy ? 0.0f : 1.0f / temperature;    // fl(1/T), IEEE division on the host
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int st = launch_gemm<3>(A, B, logits, M, N, K, bn, s, sel, RopeArgs{}, &n_tiles);
    if (st != BIV_OK) return st;
    if (rows_per_req > kMaxAcceptRows) {          // the two kernels instead
        const int st2 = launch_pdl(tile_winners_kernel, dim3((M + 7) / 8), dim3(256), 0, s,
                                   static_cast<const unsigned long long*>(workspace), M, n_tiles, tokens);
        if (st2 != BIV_OK) return st2;
        return biv_verify_accept(tokens, draft, p0, n_req, rows_per_req, accept_len, new_len, stream);
    }
    // one warp per row of the request (up to 32 warps)
    const int warps = std::min(32, std::max(1, rows_per_req));
    return launch_pdl(winners_accept_kernel, dim3(static_cast<unsigned>(n_req)), dim3(32 * warps),
                      static_cast<size_t>(rows_per_req) * sizeof(int32_t), s,
                      static_cast<const unsigned long long*>(workspace), n_tiles, tokens, draft, p0, rows_per_req,
                      accept_len, new_len);
}

extern "C" int biv_rope_pack_qkv_weights(const void* w_qkv, void* w_packed, int Hq, int Hkv, int hd, int K,
                                         biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (Hq <= 0 || Hkv <= 0 || hd <= 0 || hd % 16 != 0 || hd > 256 || K <= 0 || K % 8 != 0) return BIV_ERR_SHAPE;
    if (!w_qkv || !w_packed) return BIV_ERR_NULL;
    if (!aligned16(w_qkv) || !aligned16(w_packed)) return BIV_ERR_ALIGN;
    if (w_qkv == w_packed) return BIV_ERR_VALUE;
    // no early trigger: a GEMM launched right after reads these weights
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((Hq + 2 * Hkv) * hd));
    cfg.blockDim = dim3(128);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    return cuda_status(cudaLaunchKernelEx(&cfg, rope_pack_kernel, static_cast<const __nv_bfloat16*>(w_qkv),
                                          static_cast<__nv_bfloat16*>(w_packed), Hq, Hkv, hd, K));
}

extern "C" int biv_gemm_qkv_rope(const void* A, const void* B_packed, void* q_out, void* k_cache, void* v_cache,
                                 void* qkv_out, const int32_t* row_slot, const int32_t* row_pos,
                                 const int32_t* rows_keep, int W, int K, int d, int Hq, int Hkv, int hd, int n_slots,
                                 int max_len, float theta, biv_stream_t stream) {
    BIV_TRACE_CALL();
    if (W < 0 || K < 1 || d <= 0 || d % 8 != 0 || Hq <= 0 || Hkv <= 0 || hd <= 0 || hd % 16 != 0 || hd > 256 ||
        n_slots <= 0 || max_len <= 0 || Hq % Hkv != 0)
        return BIV_ERR_SHAPE;
    if (W % K != 0) return BIV_ERR_SHAPE;
    if (!(theta > 1.0f) || !std::isfinite(theta)) return BIV_ERR_VALUE;
    if (W == 0) return BIV_OK;
    if (!A || !B_packed || !q_out || !k_cache || !v_cache || !row_slot || !row_pos) return BIV_ERR_NULL;
    if (!aligned16(A) || !aligned16(B_packed) || !aligned16(q_out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (qkv_out && !aligned16(qkv_out)))
        return BIV_ERR_ALIGN;
    const int N = (Hq + 2 * Hkv) * hd;
    RopeArgs rp;
    rp.q_out = static_cast<__nv_bfloat16*>(q_out);
    rp.kc = static_cast<__nv_bfloat16*>(k_cache);
    rp.vc = static_cast<__nv_bfloat16*>(v_cache);
    rp.qkv_out = static_cast<__nv_bfloat16*>(qkv_out);
    rp.row_slot = row_slot;
    rp.row_pos = row_pos;
    rp.rows_keep = rows_keep;
    rp.Hq = Hq;
    rp.Hkv = Hkv;
    rp.hd = hd;
    rp.n_slots = n_slots;
    rp.max_len = max_len;
    rp.K = K;
    rp.theta = theta;
    return launch_gemm<4>(A, B_packed, nullptr, W, N, d, biv_gemm_tile_n(W, N, d), reinterpret_cast<cudaStream_t>(stream),
                          SelectArgs{}, rp);
}
