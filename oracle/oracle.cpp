// CPU oracle for the batch-invariant verification step.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
// baseline leg use it.  It shares no code, header, table or constant
// generator with the CUDA library.
//
// Plain, slow, obviously correct: one loop nest per definition, fp64
// arithmetic for RMSNorm / GEMM / attention / RoPE / SwiGLU, and the exact
// fp32 selection rule (Philox4x32-10 counter noise, own fp32 log, key,
// lowest-index argmax) for Gumbel-max.  Rows are independent, so loops over
// rows may run in parallel (OpenMP) without changing any result.
//
// Sources (pages are cited by title and paragraph):
//   [DVR]      tgstat @ashnskt post 392 -- batch-invariant kernels (para 1),
//              LLM-42 Decode-Verify-Rollback (paras 3-4: fixed-batch verifier,
//              anchor at the last correct token, KV overwrite, W = N*K).
//   [GUIDE]    "NVIDIA publishes AI inference guide, 6x lossless speedup":
//              speculative decoding (verify the drafts, restart at the break
//              point), GQA tile rule G*(1+D) <= 128.
//   [COUPLING] tginsight AIexTime post 185, "Coupling without Communication
//              and Drafter-Invariant Speculative Decoding": Gumbel-max
//              sampling, shared noise for drafter and target, compare tokens.
//   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
//              as easy as 1, 2, 3", SC'11.
//
// Readings where the pages are silent (each is listed in the design notes):
// RMSNorm keeps eps inside the root; GQA maps query head h to KV head
// h / (Hq/Hkv); RoPE is the rotate-half form; the FFN is SwiGLU with the gate
// rows first; noise counter = (v >> 2, pos, req, 0) with key = seed, word
// v & 3; uniform u = (2*(w >> 9) + 1) * 2^-24; the log is the routine below;
// key = fl(fl(x * fl(1/T)) + g); ties go to the lowest index; T = 0 is greedy.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double bf16_to_double(uint16_t h) {
    uint32_t u = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return static_cast<double>(f);
}

// Round a double to the nearest bf16, ties to even.  The fp64 -> fp32 step
// rounds to odd (truncate, then set the last bit if inexact), which makes the
// following fp32 -> bf16 round-to-nearest-even step exact-once rounding.
uint16_t double_to_bf16(double x) {
    if (std::isnan(x)) return 0x7fc0;
    float f = static_cast<float>(x);
    uint32_t u;
    if (std::isfinite(f) && static_cast<double>(f) != x) {
        if (std::fabs(static_cast<double>(f)) > std::fabs(x)) f = std::nextafter(f, 0.0f);
        std::memcpy(&u, &f, 4);
        u |= 1u;
    } else {
        std::memcpy(&u, &f, 4);
    }
    uint32_t lsb = (u >> 16) & 1u;
    uint32_t r = u + 0x7fffu + lsb;
    return static_cast<uint16_t>(r >> 16);
}

float bits_to_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t float_to_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

}  // namespace

extern "C" {

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

// ---------------------------------------------------------------- bf16 I/O
void orc_bf16_to_f64(const uint16_t* x, long long n, double* y) {
    for (long long i = 0; i < n; ++i) y[i] = bf16_to_double(x[i]);
}

void orc_f64_to_bf16(const double* x, long long n, uint16_t* y) {
    for (long long i = 0; i < n; ++i) y[i] = double_to_bf16(x[i]);
}

// ------------------------------------------------------------------ RMSNorm
// [DVR] para 1 names RMSNorm among the kernels made batch-invariant.
// y[r][i] = x[r][i] / sqrt(mean_i x[r][i]^2 + eps) * w[i], in fp64.
void orc_rmsnorm(const double* x, const double* w, int rows, int d, double eps, double* y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        const double* xr = x + (long long)r * d;
        double ss = 0.0;
        for (int i = 0; i < d; ++i) ss += xr[i] * xr[i];
        double inv = 1.0 / std::sqrt(ss / d + eps);
        for (int i = 0; i < d; ++i) y[(long long)r * d + i] = xr[i] * inv * w[i];
    }
}

// --------------------------------------------------------------------- GEMM
// [DVR] para 1: the matmul whose K dimension must never be split.  The
// definition itself: C[m][n] = sum_k A[m][k] * B[n][k], with B a bf16 weight
// in nn.Linear layout [N, K].  Products of bf16 values are exact in fp64.
void orc_gemm(const double* A, const uint16_t* B, int M, int N, int K, double* C) {
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        const uint16_t* b = B + (long long)n * K;
        std::vector<double> bd(K);
        for (int k = 0; k < K; ++k) bd[k] = bf16_to_double(b[k]);
        for (int m = 0; m < M; ++m) {
            const double* a = A + (long long)m * K;
            double s = 0.0;
            for (int k = 0; k < K; ++k) s += a[k] * bd[k];
            C[(long long)m * N + n] = s;
        }
    }
}

// Single output elements C[m][n] for sampled (m, n) pairs (full-size checks).
void orc_gemm_sampled(const uint16_t* A, const uint16_t* B, int K, const long long* m_idx,
                      const long long* n_idx, int count, double* out) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < count; ++i) {
        const uint16_t* a = A + m_idx[i] * K;
        const uint16_t* b = B + n_idx[i] * K;
        double s = 0.0;
        for (int k = 0; k < K; ++k) s += bf16_to_double(a[k]) * bf16_to_double(b[k]);
        out[i] = s;
    }
}

// --------------------------------------------------------------------- RoPE
// Rotate-half rotary embedding at absolute position pos (Llama reading; the
// pages do not describe the model).  x: [rows, heads, hd], rotated in place.
void orc_rope(double* x, const int* row_pos, int rows, int heads, int hd, double theta) {
    int half = hd / 2;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < heads; ++h) {
            double* v = x + ((long long)r * heads + h) * hd;
            for (int i = 0; i < half; ++i) {
                double freq = std::pow(theta, -2.0 * i / hd);
                double ang = row_pos[r] * freq;
                double c = std::cos(ang), s = std::sin(ang);
                double a = v[i], b = v[i + half];
                v[i] = a * c - b * s;
                v[i + half] = b * c + a * s;
            }
        }
    }
}

// --------------------------------------------------------------- attention
// Decode attention of each verify row over its own cache prefix [0, pos]
// ([DVR] para 3: each verified token attends to everything before it, with
// the window's own rows already written to the cache).  Exact softmax in
// fp64, no splitting (the split/combine of the GPU path is an identity).
// q: [W, Hq, hd]; caches: [n_slots, Hkv, max_len, hd] bf16; o: [W, Hq, hd].
void orc_attention(const double* q, const uint16_t* kc, const uint16_t* vc, const int* row_slot,
                   const int* row_pos, int W, int Hq, int Hkv, int hd, int n_slots, int max_len,
                   double* o) {
    int G = Hq / Hkv;
    double scale = 1.0 / std::sqrt((double)hd);
    (void)n_slots;
#pragma omp parallel for schedule(dynamic)
    for (int w = 0; w < W; ++w) {
        int p = row_pos[w];
        std::vector<double> s(p + 1);
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / G;
            const double* qv = q + ((long long)w * Hq + h) * hd;
            long long base = ((long long)row_slot[w] * Hkv + kvh) * max_len;
            double mx = -INFINITY;
            for (int j = 0; j <= p; ++j) {
                const uint16_t* kj = kc + (base + j) * hd;
                double dot = 0.0;
                for (int t = 0; t < hd; ++t) dot += qv[t] * bf16_to_double(kj[t]);
                s[j] = dot * scale;
                if (s[j] > mx) mx = s[j];
            }
            double den = 0.0;
            for (int j = 0; j <= p; ++j) { s[j] = std::exp(s[j] - mx); den += s[j]; }
            double* ov = o + ((long long)w * Hq + h) * hd;
            for (int t = 0; t < hd; ++t) ov[t] = 0.0;
            for (int j = 0; j <= p; ++j) {
                const uint16_t* vj = vc + (base + j) * hd;
                double pj = s[j] / den;
                for (int t = 0; t < hd; ++t) ov[t] += pj * bf16_to_double(vj[t]);
            }
        }
    }
}

// Sampled attention outputs: only the listed (row, head) pairs.
void orc_attention_sampled(const uint16_t* q_bf16, const uint16_t* kc, const uint16_t* vc,
                           const int* row_slot, const int* row_pos, int Hq, int Hkv, int hd,
                           int max_len, const int* rows, const int* heads, int count, double* o) {
    int G = Hq / Hkv;
    double scale = 1.0 / std::sqrt((double)hd);
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < count; ++i) {
        int w = rows[i], h = heads[i], p = row_pos[w], kvh = h / G;
        const uint16_t* qv = q_bf16 + ((long long)w * Hq + h) * hd;
        long long base = ((long long)row_slot[w] * Hkv + kvh) * max_len;
        std::vector<double> s(p + 1);
        double mx = -INFINITY;
        for (int j = 0; j <= p; ++j) {
            double dot = 0.0;
            for (int t = 0; t < hd; ++t)
                dot += bf16_to_double(qv[t]) * bf16_to_double(kc[(base + j) * hd + t]);
            s[j] = dot * scale;
            if (s[j] > mx) mx = s[j];
        }
        double den = 0.0;
        for (int j = 0; j <= p; ++j) { s[j] = std::exp(s[j] - mx); den += s[j]; }
        for (int t = 0; t < hd; ++t) {
            double acc = 0.0;
            for (int j = 0; j <= p; ++j) acc += s[j] / den * bf16_to_double(vc[(base + j) * hd + t]);
            o[(long long)i * hd + t] = acc;
        }
    }
}

// ------------------------------------------------------------------ SwiGLU
// h = silu(gate) * up with silu(g) = g / (1 + exp(-g)); gu: [rows, 2F] with
// the F gate columns first.
void orc_silu_mul(const double* gu, int rows, int F, double* h) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r)
        for (int i = 0; i < F; ++i) {
            double g = gu[(long long)r * 2 * F + i], u = gu[(long long)r * 2 * F + F + i];
            h[(long long)r * F + i] = g / (1.0 + std::exp(-g)) * u;
        }
}

// ---------------------------------------------------------------- KV write
// [DVR] para 3: at every verification the fast path's cache rows are
// overwritten by the verifier's values.  Row w of the window writes its K
// and V (bf16 [W, Hkv, hd]) at (row_slot[w], position row_pos[w]).
void orc_kv_overwrite(uint16_t* kc, uint16_t* vc, const uint16_t* k_new, const uint16_t* v_new,
                      const int* row_slot, const int* row_pos, int W, int Hkv, int hd, int max_len) {
    for (int w = 0; w < W; ++w)
        for (int h = 0; h < Hkv; ++h) {
            long long dst = (((long long)row_slot[w] * Hkv + h) * max_len + row_pos[w]) * hd;
            long long src = ((long long)w * Hkv + h) * hd;
            for (int t = 0; t < hd; ++t) {
                kc[dst + t] = k_new[src + t];
                vc[dst + t] = v_new[src + t];
            }
        }
}

// ------------------------------------------------------------ Philox4x32-10
// Salmon et al., SC'11: ten rounds of the 4x32 Philox S-box; each round
// multiplies words 0 and 2 by the two round multipliers, swaps and xors the
// high halves with the other words and the round key; the key is bumped by
// the two Weyl constants between rounds.
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// Uniform in (0,1) from a 32-bit word: u = (2 * (w >> 9) + 1) * 2^-24.
// Exact in fp32; 2^23 distinct values, never 0 or 1.
float orc_uniform(uint32_t w) {
    uint32_t k = 2u * (w >> 9) + 1u;          // odd, < 2^24: exact in fp32
    return (float)k * 5.9604644775390625e-8f; // 2^-24, exact scaling
}

// Natural log of a positive normal fp32 value, built only from IEEE single
// operations (+, -, *, /, fma), so that any conforming machine gets the same
// bits.  Method: x = m * 2^e with m in [fl(sqrt 2)/2, fl(sqrt 2)); with
// f = m - 1 and s = f / (2 + f), ln m = 2 atanh(s) = 2s * sum_k s^(2k)/(2k+1)
// (series truncated after k = 6, Horner in fma); ln x = e*ln2_hi +
// (e*ln2_lo + ln m) with ln 2 split into a 17-bit head 0x1.62e4p-1 and the
// fp32-rounded remainder.
float orc_log_f32(float x) {
    uint32_t b = float_to_bits(x);
    int e = (int)((b >> 23) & 0xffu) - 127;
    uint32_t frac = b & 0x007fffffu;
    uint32_t mb = frac | 0x3f800000u;             // m in [1, 2)
    if (frac >= 0x003504f3u) {                    // m >= fl(sqrt 2): halve m
        mb -= 0x00800000u;
        e += 1;
    }
    float m = bits_to_float(mb);
    float f = m - 1.0f;                           // exact (Sterbenz)
    float t = 2.0f + f;
    float s = f / t;
    float z = s * s;
    const float c[7] = {
        bits_to_float(0x3f800000u),  // 1
        bits_to_float(0x3eaaaaabu),  // 1/3
        bits_to_float(0x3e4ccccdu),  // 1/5
        bits_to_float(0x3e124925u),  // 1/7
        bits_to_float(0x3de38e39u),  // 1/9
        bits_to_float(0x3dba2e8cu),  // 1/11
        bits_to_float(0x3d9d89d9u),  // 1/13
    };
    float p = c[6];
    for (int k = 5; k >= 0; --k) p = std::fmaf(p, z, c[k]);
    float r = s + s;
    float lnm = r * p;
    float ef = (float)e;
    const float ln2_hi = bits_to_float(0x3f317200u);  // 0x1.62e4p-1
    const float ln2_lo = bits_to_float(0x35bfbe8eu);  // fl(ln 2 - ln2_hi)
    float u = std::fmaf(ef, ln2_lo, lnm);
    return std::fmaf(ef, ln2_hi, u);
}

void orc_log_batch(const float* x, long long n, float* y) {
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < n; ++i) y[i] = orc_log_f32(x[i]);
}

// Gumbel(0,1) noise from a uniform: g = -log(-log(u)).
float orc_gumbel_from_word(uint32_t w) {
    float u = orc_uniform(w);
    float a = orc_log_f32(u);
    float t = -a;
    return -orc_log_f32(t);
}

void orc_gumbel_from_words(const uint32_t* w, long long n, float* g) {
#pragma omp parallel for schedule(static)
    for (long long i = 0; i < n; ++i) g[i] = orc_gumbel_from_word(w[i]);
}

// The noise for vocabulary entry v of the token at absolute position pos of
// request req ([COUPLING]: the noise does not depend on the logits, so it
// is a pure function of who/where/which entry).  Counter (v >> 2, pos, req, 0),
// key (seed low word, seed high word), output word v & 3.
float orc_gumbel(uint64_t seed, uint32_t req, uint32_t pos, uint32_t v) {
    uint32_t ctr[4] = {v >> 2, pos, req, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return orc_gumbel_from_word(out[v & 3u]);
}

void orc_gumbel_row(uint64_t seed, uint32_t req, uint32_t pos, int V, float* g) {
    for (int v = 0; v < V; ++v) g[v] = orc_gumbel(seed, req, pos, (uint32_t)v);
}

// ------------------------------------------------------------- selection
// [COUPLING]: add Gumbel(0,1) noise to the (temperature-scaled) logits and
// take the argmax; this samples from softmax(x / T) without a softmax.
// key_v = fl(fl(x_v * invT) + g_v), invT = fl(1/T); the largest key wins,
// the lowest index wins among equal keys, a NaN key never beats a number;
// T == 0 selects the largest logit (lowest index on ties).  Row w selects
// the token at position row_pos[w] + 1 of request row_req[w].
static bool key_beats(float k, int v, float best, int best_v) {
    // Order: NaN below everything; numbers by value (-0 == +0); ties -> lower index.
    bool kn = std::isnan(k), bn = std::isnan(best);
    if (kn && bn) return v < best_v;
    if (kn) return false;
    if (bn) return true;
    if (k > best) return true;
    if (k < best) return false;
    return v < best_v;
}

void orc_gumbel_argmax(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                       const int* row_pos, uint64_t seed, float temperature, int* tokens) {
    float invT = temperature > 0.0f ? 1.0f / temperature : 0.0f;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        const float* x = logits + (long long)r * ld;
        uint32_t pos = (uint32_t)(row_pos[r] + 1);
        float best = 0.0f;
        int best_v = -1;
        for (int v = 0; v < V; ++v) {
            float key;
            if (temperature > 0.0f) {
                float a = x[v] * invT;
                key = a + orc_gumbel(seed, row_req[r], pos, (uint32_t)v);
            } else {
                key = x[v];
            }
            if (best_v < 0 || key_beats(key, v, best, best_v)) { best = key; best_v = v; }
        }
        tokens[r] = best_v;
    }
}

// ----------------------------------------------------------- Gumbel top-k
// [COUPLING]: the Gumbel-max trick gives top-k sampling directly: the k
// entries with the largest keys, in decreasing key order, are a sample of k
// distinct tokens without replacement from softmax(x / T) (Kool, van Hoof &
// Welling, "Stochastic Beams and Where to Find Them", ICML 2019).  Same keys,
// same order (ties -> lower index, NaN keys last) as orc_gumbel_argmax, so
// column 0 is the Gumbel-max token.
void orc_gumbel_topk(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                     const int* row_pos, uint64_t seed, float temperature, int k, int* out) {
    float invT = temperature > 0.0f ? 1.0f / temperature : 0.0f;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        const float* x = logits + (long long)r * ld;
        uint32_t pos = (uint32_t)(row_pos[r] + 1);
        std::vector<float> key(V);
        std::vector<int> idx(V);
        for (int v = 0; v < V; ++v) {
            if (temperature > 0.0f) {
                float a = x[v] * invT;
                key[v] = a + orc_gumbel(seed, row_req[r], pos, (uint32_t)v);
            } else {
                key[v] = x[v];
            }
            idx[v] = v;
        }
        std::partial_sort(idx.begin(), idx.begin() + k, idx.end(),
                          [&](int a, int b) { return key_beats(key[a], a, key[b], b); });
        for (int j = 0; j < k; ++j) out[(long long)r * k + j] = idx[j];
    }
}

// ------------------------------------------------------- n-gram drafter
// Training-free n-gram lookup drafter (NVIDIA inference guide page, the
// drafting methods it lists: repeated fragments of the earlier text are found
// and copied).  Reading: for request r with committed history h[0..L) take
// the longest n in [n_min, n_max] whose last-n-token suffix also occurs
// earlier with at least one token after it; of those occurrences take the
// most recent (largest start p <= L - n - 1); the drafts copy the K tokens
// that followed it, s = p + n: d_j = e[s + j] where e is the history with the
// drafts appended (a copy that runs past the end continues from its own
// output, as an LZ77 copy does, so a periodic text is continued exactly).  No
// match for any n: all K drafts are h[L - 1] (0 for an empty history).
// draft_src[r] = s, or -1.
void orc_ngram_draft(const int* hist, int N, long long ld, const int* len, int n_max, int n_min, int K,
                     int* drafts, int* draft_src) {
    for (int r = 0; r < N; ++r) {
        const int* h = hist + (long long)r * ld;
        const int L = len[r];
        int src = -1;
        for (int n = n_max; n >= n_min && src < 0; --n) {
            if (L < n + 1) continue;
            for (int p = L - n - 1; p >= 0; --p) {
                bool match = true;
                for (int i = 0; i < n; ++i) {
                    if (h[p + i] != h[L - n + i]) { match = false; break; }
                }
                if (match) { src = p + n; break; }
            }
        }
        draft_src[r] = src;
        int* d = drafts + (long long)r * K;
        for (int j = 0; j < K; ++j) {
            if (src < 0) {
                d[j] = L > 0 ? h[L - 1] : 0;
            } else {
                const int t = src + j;
                d[j] = t < L ? h[t] : d[t - L];
            }
        }
    }
}

// --------------------------------------------------------------- accept
// [COUPLING] + [GUIDE]: with shared noise the verifier compares tokens only.
// Row j of request r outputs y_{j+1}; draft[r*K + j] holds d_{j+1}.  The
// accepted length is the index of the first mismatch plus one (K if none):
// y_1..y_L are emitted, all of them the target's own tokens, and request r
// rolls back to new_len = p0 + L ([DVR] para 3).
void orc_verify_accept(const int* target, const int* draft, const int* p0, int N, int K,
                       int* accept_len, int* new_len) {
    for (int r = 0; r < N; ++r) {
        int L = K;
        for (int j = 0; j < K; ++j) {
            if (target[r * K + j] != draft[r * K + j]) { L = j + 1; break; }
        }
        accept_len[r] = L;
        new_len[r] = p0[r] + L;
    }
}

// --------------------------------------------------------------- GQA tile
// [GUIDE] GQA tile rule: the G query heads of one KV head times the 1 + D
// verified rows must fit one tile: G * (1 + D) <= tile, so D = tile / G - 1.
int orc_gqa_max_drafts(int G, int tile) {
    if (G <= 0 || tile < G) return -1;
    return tile / G - 1;
}

}  // extern "C"
