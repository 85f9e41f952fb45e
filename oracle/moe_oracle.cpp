// CPU oracle for the MoE expert layer.  TEST INFRASTRUCTURE ONLY: the tests,
// the smoke check and the CPU-baseline leg of the benchmark call it; the
// product path never does.  It shares no code, header or table with the CUDA
// library and is built on its own (g++, -ffp-contract=off).
//
// Each function is the plain definition of one step, written as plain loops
// in the order the sources describe the layer:
//   * "Mixture of Experts in transformers" -- MoE basics (a router picks k of
//     E experts per token) and pluggable expert backends (grouped_mm sorts the
//     tokens by expert id and runs one grouped GEMM; eager loops the experts);
//   * "Hugging Face Transformers: MoE and FP8 kernel optimisation"
//     (transformers PR #45621) -- section 1 (fine-grained FP8 entries:
//     fp8_act_quant / per_token_cast_to_fp8, grouped_fp8_matmul), section 2
//     (sentinel slots are left out of the histogram / sorted last, and the
//     per-expert offsets end at the number of live rows), section 3 (outputs
//     of sentinel rows must not be left uninitialised);
//   * "LlamaFactory Triton fused MoE kernel" (LlamaFactory PR #10481) --
//     section 1: scatter, grouped GEMM fc1, silu(gate)*up, grouped GEMM fc2,
//     gather.
//
// Precision: bf16 operands are widened exactly to fp32; dot products, SwiGLU
// and the combine accumulate in double and are stored as fp32.  FP8
// quantisation is done in fp32 (amax, two IEEE divides, one rounding to
// e4m3) because that arithmetic decides the bytes.
//
// Threads: the loops over independent rows carry OpenMP pragmas.  The
// default build (no -fopenmp) ignores them and runs on one core; the timing
// build of the CPU baseline adds -fopenmp and runs the rows in parallel.  Each
// output element is computed by one thread in the same order either way, so
// the two builds agree bit for bit (a CPU test checks that).
//
// Parity pins (all in the CPU test-suite): e4m3 codec against torch's
// float8_e4m3fn and the format definition; bf16 rounding against torch's
// float32 -> bfloat16 conversion on every upper half and hand-worked ties;
// top-k and the stable sort against brute force; quantisation against exact
// special cases; the permute of e4m3 rows and their scale rows against numpy
// indexing by token; the bf16 layer against a float64 per-token expert loop
// and a dense SwiGLU MLP (E = 1, k = 1); the FP8 layer against a float64
// per-token loop with torch's codecs.

#include <algorithm>
#include <cmath>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

inline float bf16_to_f32(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

inline uint16_t f32_to_bf16_rne(float f) {
    if (std::isnan(f)) return 0x7FC0;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return static_cast<uint16_t>(u >> 16);
}

// ---------------------------------------------------------------------------
// OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
// infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448; normals
// down to 2^-6; subnormals m/8 * 2^-6, m = 1..7.

const float kE4M3Max = 448.0f;

float e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return std::nanf("");
    double v = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
    return static_cast<float>(s ? -v : v);
}

// Round to nearest, ties to even mantissa, saturating to +-448 (no overflow
// to NaN).  Every scaling below is by a power of two, so it is exact in fp32
// and the only rounding is the rint() to an integer mantissa.
uint8_t e4m3_encode(float v) {
    if (std::isnan(v)) return 0x7F;
    uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
    float a = std::fabs(v);
    if (a >= kE4M3Max) return sign | 0x7E;
    if (a < 0x1p-6f) {                    // subnormal grid, spacing 2^-9
        float m = std::nearbyint(a * 512.0f);          // 0..8
        return sign | static_cast<uint8_t>(m);         // m == 8 is 2^-6 (code 0x08)
    }
    int ex;
    std::frexp(a, &ex);                   // a = f * 2^ex, f in [0.5, 1)
    int eu = ex - 1;                      // a in [2^eu, 2^(eu+1))
    float m = std::nearbyint(std::ldexp(a, 3 - eu));   // in [8, 16]
    if (m == 16.0f) { m = 8.0f; eu += 1; }
    if (eu > 8) return sign | 0x7E;       // unreachable for a < 448
    return sign | static_cast<uint8_t>(((eu + 7) << 3) | (static_cast<int>(m) - 8));
}

// The 256 decoded values, filled once from e4m3_decode (same values; only
// saves re-deriving them inside the GEMM loops).
const float* e4m3_table() {
    static float table[256];
    static bool ready = [] {
        for (int c = 0; c < 256; ++c) table[c] = e4m3_decode(static_cast<uint8_t>(c));
        return true;
    }();
    (void)ready;
    return table;
}

// amax / 448 in fp32; a group or block of zeros gets scale 1.
inline float fp8_scale_from_amax(float amax) {
    return amax == 0.0f ? 1.0f : amax / kE4M3Max;
}

}  // namespace

extern "C" {

// Threads the row loops run on: 1 in the default build.
int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// ---------------------------------------------------------------- e4m3 codec
void orc_e4m3_encode(const float* v, int64_t n, uint8_t* q) {
    for (int64_t i = 0; i < n; ++i) q[i] = e4m3_encode(v[i]);
}

void orc_e4m3_decode(const uint8_t* q, int64_t n, float* v) {
    for (int64_t i = 0; i < n; ++i) v[i] = e4m3_decode(q[i]);
}

void orc_bf16_round(const float* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(v[i]);
}

// ---------------------------------------------------------------- routing
// Top-k routing ("MoE basics": the router picks a small subset of the E
// experts for each token).  l'[t,e] = logits[t,e] + bias[e] (fp32 add; no add
// without a bias).  The k experts are picked by k rounds of arg-max over l',
// ties to the lower expert id; slot j holds the j-th pick.  Weights are the
// softmax over the k picked l' (renormalize != 0) or the full softmax over all
// E evaluated at the picks (renormalize == 0), in double, stored fp32.
void orc_route_topk(const float* logits, const float* bias, int T, int E, int k,
                    int renormalize, int32_t* ids, float* w) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        std::vector<float> lp(E);
        std::vector<char> taken(E);
        for (int e = 0; e < E; ++e)
            lp[e] = bias ? logits[(int64_t)t * E + e] + bias[e] : logits[(int64_t)t * E + e];
        std::fill(taken.begin(), taken.end(), 0);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || lp[e] > lp[best]) best = e;   // strict: ties keep the lower id
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        double mx = lp[ids[(int64_t)t * k]];
        double den = 0.0;
        if (renormalize) {
            for (int j = 0; j < k; ++j) den += std::exp((double)lp[ids[(int64_t)t * k + j]] - mx);
        } else {
            for (int e = 0; e < E; ++e) den += std::exp((double)lp[e] - mx);
        }
        for (int j = 0; j < k; ++j)
            w[(int64_t)t * k + j] =
                static_cast<float>(std::exp((double)lp[ids[(int64_t)t * k + j]] - mx) / den);
    }
}

// Sentinel marking: a slot flagged in mask becomes unrouted, expert id = E.
void orc_mark_sentinels(int32_t* ids, const uint8_t* mask, int64_t R, int E) {
    for (int64_t i = 0; i < R; ++i)
        if (mask[i]) ids[i] = E;
}

// Sort by expert id (section 2 of the transformers write-up; grouped_mm
// backend of "MoE in transformers").  Slots are flat indices f = t*k + j with
// key ids[f] in [0, E]; id E is the sentinel, which sorts last.  A stable sort
// on the key gives sorted_rows (ties by flat index, i.e. by token);
// row_pos is its inverse.  offsets[0] = 0 and offsets[e+1] = offsets[e] +
// #{f : ids[f] == e} for e < E -- the sentinel bin is left out, so
// offsets[E] is the number of live rows.
void orc_sort_by_expert(const int32_t* ids, int64_t R, int E, int32_t* sorted_rows,
                        int32_t* row_pos, int32_t* offsets) {
    std::vector<int32_t> order(R);
    for (int64_t f = 0; f < R; ++f) order[f] = static_cast<int32_t>(f);
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return ids[a] < ids[b]; });
    for (int64_t p = 0; p < R; ++p) {
        sorted_rows[p] = order[p];
        row_pos[order[p]] = static_cast<int32_t>(p);
    }
    std::vector<int64_t> cnt(E, 0);
    for (int64_t f = 0; f < R; ++f)
        if (ids[f] >= 0 && ids[f] < E) cnt[ids[f]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = static_cast<int32_t>(offsets[e] + cnt[e]);
}

// Expert parallelism ("Mixture of Experts in transformers", expert
// parallelism): the experts are sharded on their first dimension, rank r
// holding the global experts [first, first + E_local); a router pick of a
// local expert becomes its local id (id - first), any other pick -- another
// rank's expert, or the global sentinel E_global -- becomes the local
// sentinel E_local, so the local layer leaves it out (section 2 of the
// transformers MoE/FP8 write-up).  An id outside [0, E_global] is not a pick
// at all and becomes the sentinel too.
void orc_ep_local_ids(const int32_t* ids, int64_t R, int E_global, int first, int E_local,
                      int32_t* local_ids) {
    for (int64_t i = 0; i < R; ++i) {
        const int32_t id = ids[i];
        local_ids[i] = (id >= first && id < first + E_local && id < E_global) ? id - first : E_local;
    }
}

// ---------------------------------------------------------------- FP8 quant
// Per-token activation quantisation (fp8_act_quant / per_token_cast_to_fp8
// of section 1): for row m and 128-column group g,
//   s[m,g] = amax/448 (1 if amax = 0),  q[m,c] = e4m3(x[m,c] / s[m,g]).
// x is bf16 [M, K], K a multiple of 128; q is [M, K]; s is fp32 [M, K/128].
void orc_quant_act_fp8(const uint16_t* x, int64_t M, int K, uint8_t* q, float* s) {
    const int G = K / 128;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int g = 0; g < G; ++g) {
            const uint16_t* xr = x + m * K + g * 128;
            float amax = 0.0f;
            for (int c = 0; c < 128; ++c) amax = std::max(amax, std::fabs(bf16_to_f32(xr[c])));
            float sc = fp8_scale_from_amax(amax);
            s[m * G + g] = sc;
            for (int c = 0; c < 128; ++c) q[m * K + g * 128 + c] = e4m3_encode(bf16_to_f32(xr[c]) / sc);
        }
    }
}

// Block weight quantisation: e4m3 weights with one fp32 scale per 128x128
// block (the fine-grained FP8 weight format of section 1).  W bf16 [E, N, K],
// K a multiple of 128, N any (the last row block may be short);
// s is [E, ceil(N/128), K/128].
void orc_quant_weight_fp8(const uint16_t* W, int E, int N, int K, uint8_t* q, float* s) {
    const int NB = (N + 127) / 128, KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int e = 0; e < E; ++e) {
        for (int nb = 0; nb < NB; ++nb) {
            const uint16_t* We = W + (int64_t)e * N * K;
            uint8_t* qe = q + (int64_t)e * N * K;
            const int n1 = std::min(N, nb * 128 + 128);
            for (int kb = 0; kb < KB; ++kb) {
                float amax = 0.0f;
                for (int n = nb * 128; n < n1; ++n)
                    for (int c = kb * 128; c < kb * 128 + 128; ++c)
                        amax = std::max(amax, std::fabs(bf16_to_f32(We[(int64_t)n * K + c])));
                float sc = fp8_scale_from_amax(amax);
                s[((int64_t)e * NB + nb) * KB + kb] = sc;
                for (int n = nb * 128; n < n1; ++n)
                    for (int c = kb * 128; c < kb * 128 + 128; ++c)
                        qe[(int64_t)n * K + c] = e4m3_encode(bf16_to_f32(We[(int64_t)n * K + c]) / sc);
            }
        }
    }
}

// ---------------------------------------------------------------- permute
// Scatter (moe_scatter of the LlamaFactory write-up): xp[p] = x[sorted_rows[p] / k]
// for p < L = offsets[E]; rows p >= L are left as they are.  elem_bytes is 2
// for bf16 rows and 1 for e4m3 rows.  With scales (FP8) the per-group scale
// rows follow the same map: xs[p, :] = s[sorted_rows[p] / k, :].
void orc_permute(const void* x, const float* x_scales, int elem_bytes, int64_t T, int H, int k,
                 const int32_t* sorted_rows, int64_t L, void* xp, float* xp_scales) {
    const int G = H / 128;
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < L; ++p) {
        int64_t t = sorted_rows[p] / k;
        std::memcpy(static_cast<char*>(xp) + p * H * elem_bytes,
                    static_cast<const char*>(x) + t * H * elem_bytes, (size_t)H * elem_bytes);
        if (x_scales && xp_scales)
            for (int g = 0; g < G; ++g) xp_scales[p * G + g] = x_scales[t * G + g];
    }
    (void)T;
}

// ---------------------------------------------------------------- grouped GEMM
// Grouped GEMM (group_gemm_same_nk of the LlamaFactory write-up; grouped_mm
// backend): for every expert e and row p in [offsets[e], offsets[e+1]),
//   C[p, n] = sum_c A[p, c] * B[e, n, c]      (B is [E, N, K], K contiguous)
// Rows at or beyond offsets[E] are sentinel rows and come out as exact zeros
// (section 3 of the transformers write-up).  rows/n_rows (optional) restrict
// the output to the listed rows: C is then [n_rows, N].
static int expert_of_row(const int32_t* offsets, int E, int64_t p) {
    for (int e = 0; e < E; ++e)
        if (p >= offsets[e] && p < offsets[e + 1]) return e;
    return -1;
}

void orc_grouped_gemm_bf16(const uint16_t* A, const uint16_t* B, const int32_t* offsets, int E,
                           int64_t M_cap, int N, int K, const int32_t* rows, int64_t n_rows,
                           float* C) {
    int64_t nout = rows ? n_rows : M_cap;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < nout; ++i) {
        int64_t p = rows ? rows[i] : i;
        float* Ci = C + i * N;
        int e = expert_of_row(offsets, E, p);
        if (e < 0) {
            for (int n = 0; n < N; ++n) Ci[n] = 0.0f;
            continue;
        }
        std::vector<float> a(K);
        for (int c = 0; c < K; ++c) a[c] = bf16_to_f32(A[p * K + c]);
        const uint16_t* Be = B + (int64_t)e * N * K;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += (double)a[c] * (double)bf16_to_f32(Be[(int64_t)n * K + c]);
            Ci[n] = static_cast<float>(acc);
        }
    }
}

// Gradients of the bf16 grouped GEMM C[p, n] = sum_c A[p, c] B[e, n, c]
// (rows p of expert e), for training ("Mixture of Experts in transformers",
// MoE training with grouped GEMMs; section 3 of the transformers MoE/FP8
// write-up: gradients of sentinel rows must be written, as zeros).  Given the
// output gradient dC [M_cap, N] (bf16), plain chain rule, fp64 accumulation:
//   dA[p, c] = sum_n dC[p, n] * B[e, n, c]   (rows p >= offsets[E]: 0)
// With rows (n_rows > 0), only dA[rows[i], :] is computed, into dA[i * K ..).
void orc_grouped_gemm_dgrad_bf16(const uint16_t* dC, const uint16_t* B, const int32_t* offsets, int E,
                                 int64_t M_cap, int N, int K, const int32_t* rows, int64_t n_rows,
                                 float* dA) {
    const int64_t nout = rows ? n_rows : M_cap;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < nout; ++i) {
        const int64_t p = rows ? rows[i] : i;
        float* dAp = dA + i * K;
        const int e = expert_of_row(offsets, E, p);
        if (e < 0) {
            for (int c = 0; c < K; ++c) dAp[c] = 0.0f;
            continue;
        }
        std::vector<double> acc(K, 0.0);
        const uint16_t* Be = B + (int64_t)e * N * K;
        for (int n = 0; n < N; ++n) {
            const double g = bf16_to_f32(dC[p * N + n]);
            for (int c = 0; c < K; ++c) acc[c] += g * (double)bf16_to_f32(Be[(int64_t)n * K + c]);
        }
        for (int c = 0; c < K; ++c) dAp[c] = static_cast<float>(acc[c]);
    }
}

//   dB[e, n, c] = sum over rows p of expert e of dC[p, n] * A[p, c]
// (an expert without rows gets a zero gradient).  With pairs (n_pairs > 0),
// only the rows dB[pairs[2i], pairs[2i+1], :] are computed, into
// dB[i * K .. i * K + K).
void orc_grouped_gemm_wgrad_bf16(const uint16_t* A, const uint16_t* dC, const int32_t* offsets, int E,
                                 int64_t M_cap, int N, int K, const int32_t* pairs, int64_t n_pairs,
                                 float* dB) {
    (void)M_cap;
    const int64_t nout = pairs ? n_pairs : (int64_t)E * N;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < nout; ++i) {
        const int e = pairs ? pairs[2 * i] : (int)(i / N);
        const int n = pairs ? pairs[2 * i + 1] : (int)(i % N);
        std::vector<double> acc(K, 0.0);
        for (int64_t p = offsets[e]; p < offsets[e + 1]; ++p) {
            const double g = bf16_to_f32(dC[p * N + n]);
            for (int c = 0; c < K; ++c) acc[c] += g * (double)bf16_to_f32(A[p * K + c]);
        }
        for (int c = 0; c < K; ++c) dB[i * K + c] = static_cast<float>(acc[c]);
    }
}

// FP8 grouped GEMM (grouped_fp8_matmul of section 1): A is e4m3 [M_cap, K]
// with per-row, per-128-column scales sa [M_cap, K/128]; B is e4m3 [E, N, K]
// with per-128x128-block scales sb [E, ceil(N/128), K/128].
//   C[p, n] = sum_kb sa[p,kb] * sb[e, n/128, kb] * sum_{c in kb} dec(qa[p,c]) * dec(qb[e,n,c])
void orc_grouped_gemm_fp8(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                          const int32_t* offsets, int E, int64_t M_cap, int N, int K,
                          const int32_t* rows, int64_t n_rows, float* C) {
    const int KB = K / 128, NB = (N + 127) / 128;
    int64_t nout = rows ? n_rows : M_cap;
    const float* dec = e4m3_table();
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < nout; ++i) {
        int64_t p = rows ? rows[i] : i;
        float* Ci = C + i * N;
        int e = expert_of_row(offsets, E, p);
        if (e < 0) {
            for (int n = 0; n < N; ++n) Ci[n] = 0.0f;
            continue;
        }
        std::vector<float> a(K);
        for (int c = 0; c < K; ++c) a[c] = dec[qa[p * K + c]];
        const uint8_t* Be = qb + (int64_t)e * N * K;
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int kb = 0; kb < KB; ++kb) {
                double part = 0.0;
                for (int c = kb * 128; c < kb * 128 + 128; ++c)
                    part += (double)a[c] * (double)dec[Be[(int64_t)n * K + c]];
                acc += (double)sa[p * KB + kb] * (double)sb[((int64_t)e * NB + n / 128) * KB + kb] * part;
            }
            Ci[n] = static_cast<float>(acc);
        }
    }
}

// Batched expert products (the batched_mm backend of "MoE in transformers"'s
// pluggable expert backends; batched_fp8_matmul of section 1 of the
// transformers write-up): for every slot f = t*k + j whose expert e =
// ids[f] is not the sentinel E,
//   out[f, n] = sum_c x[t, c] * W[e, n, c]
// (bf16: exact widening, double accumulation; FP8: e4m3 with per-row scales
// xs [T, K/128] and block scales Ws [E, ceil(N/128), K/128], the
// block-scaled sum of orc_grouped_gemm_fp8); sentinel slots get zero rows.
// out is fp32 [T*k, N].
void orc_batched_matmul(int fp8, const void* x, const float* xs, const int32_t* ids, int64_t T, int k, int E,
                        const void* W, const float* Ws, int N, int K, float* out) {
    const int KB = K / 128, NB = (N + 127) / 128;
    const float* dec = e4m3_table();
    for (int64_t f = 0; f < T * k; ++f) {
        const int64_t t = f / k;
        const int e = ids[f];
        float* o = out + f * N;
        if (e < 0 || e >= E) {
            for (int n = 0; n < N; ++n) o[n] = 0.0f;
            continue;
        }
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            if (!fp8) {
                const uint16_t* xr = static_cast<const uint16_t*>(x) + t * K;
                const uint16_t* wr = static_cast<const uint16_t*>(W) + ((int64_t)e * N + n) * K;
                for (int c = 0; c < K; ++c) acc += (double)bf16_to_f32(xr[c]) * (double)bf16_to_f32(wr[c]);
            } else {
                const uint8_t* xr = static_cast<const uint8_t*>(x) + t * K;
                const uint8_t* wr = static_cast<const uint8_t*>(W) + ((int64_t)e * N + n) * K;
                for (int kb = 0; kb < KB; ++kb) {
                    double part = 0.0;
                    for (int c = kb * 128; c < kb * 128 + 128; ++c) part += (double)dec[xr[c]] * (double)dec[wr[c]];
                    acc += (double)xs[t * KB + kb] * (double)Ws[((int64_t)e * NB + n / 128) * KB + kb] * part;
                }
            }
            o[n] = static_cast<float>(acc);
        }
    }
}

// ---------------------------------------------------------------- SwiGLU
// silu(gate) * up on the gate_up output (LlamaFactory write-up, section 1):
// gate = Y1[p, :I] (first half of W1's rows), up = Y1[p, I:].  Rows at or
// beyond L are zero.
void orc_swiglu(const float* Y1, int64_t M_cap, int I, int64_t L, float* h) {
#pragma omp parallel for schedule(static)
    for (int64_t p = 0; p < M_cap; ++p) {
        for (int n = 0; n < I; ++n) {
            if (p >= L) { h[p * I + n] = 0.0f; continue; }
            double g = Y1[p * 2 * I + n], u = Y1[p * 2 * I + I + n];
            h[p * I + n] = static_cast<float>(g / (1.0 + std::exp(-g)) * u);
        }
    }
}

// ---------------------------------------------------------------- combine
// Weighted gather back to token order (moe_gather of the LlamaFactory
// write-up; the partial-output sum of expert parallelism in "MoE in
// transformers"):  out[t, :] = sum_{j : ids[t,j] != E} w[t,j] * Y2[row_pos[t*k+j], :]
// in j order.  A token whose slots are all sentinels gets a zero row.
void orc_combine(const float* Y2, const int32_t* ids, const float* w, const int32_t* row_pos,
                 int64_t T, int k, int H, int E, float* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        std::vector<double> acc(H, 0.0);
        for (int j = 0; j < k; ++j) {
            int64_t f = t * k + j;
            if (ids[f] == E) continue;
            const float* y = Y2 + (int64_t)row_pos[f] * H;
            for (int c = 0; c < H; ++c) acc[c] += (double)w[f] * (double)y[c];
        }
        for (int c = 0; c < H; ++c) out[t * H + c] = static_cast<float>(acc[c]);
    }
}

// ---------------------------------------------------------------- the layer
// The whole expert layer in the order of the LlamaFactory pipeline:
// route -> sentinels -> sort -> [quantise x] -> scatter -> grouped GEMM gate_up
// -> silu*up -> [bf16 round, quantise h] -> grouped GEMM down -> weighted gather.
// fp8 == 0: W1 bf16 [E, 2I, H], W2 bf16 [E, H, I].
// fp8 == 1: W1 e4m3 + scales [E, 2I/128, H/128], W2 e4m3 + scales [E, ceil(H/128), I/128].
// logits == NULL: ids/w are inputs (after any sentinel marking); otherwise they
// are outputs.  sentinel_mask may be NULL.  out is fp32 [T, H].
// Optional taps (may be NULL): sorted_rows/row_pos [T*k], offsets [E+1].
int orc_moe_forward(int fp8, const float* logits, const float* bias, const uint8_t* sentinel_mask,
                    int32_t* ids, float* w, int64_t T, int E, int k, int H, int I, int renormalize,
                    const uint16_t* x, const void* W1, const float* W1s, const void* W2,
                    const float* W2s, float* out, int32_t* sorted_rows_tap, int32_t* row_pos_tap,
                    int32_t* offsets_tap) {
    const int64_t R = T * k;
    if (logits) orc_route_topk(logits, bias, (int)T, E, k, renormalize, ids, w);
    if (sentinel_mask) orc_mark_sentinels(ids, sentinel_mask, R, E);
    std::vector<int32_t> sorted_rows(R), row_pos(R), offsets(E + 1);
    orc_sort_by_expert(ids, R, E, sorted_rows.data(), row_pos.data(), offsets.data());
    const int64_t L = offsets[E];
    std::vector<float> Y1(R * 2 * I), h(R * I), Y2(R * H);
    if (!fp8) {
        std::vector<uint16_t> xp(R * H, 0);
        orc_permute(x, nullptr, 2, T, H, k, sorted_rows.data(), L, xp.data(), nullptr);
        orc_grouped_gemm_bf16(xp.data(), static_cast<const uint16_t*>(W1), offsets.data(), E, R,
                              2 * I, H, nullptr, 0, Y1.data());
        orc_swiglu(Y1.data(), R, I, L, h.data());
        // the plain definition keeps h in fp32; the down GEMM reads it directly
#pragma omp parallel for schedule(dynamic, 4)
        for (int64_t p = 0; p < R; ++p) {
            int e = expert_of_row(offsets.data(), E, p);
            float* y = Y2.data() + p * H;
            if (e < 0) { std::fill(y, y + H, 0.0f); continue; }
            const uint16_t* We = static_cast<const uint16_t*>(W2) + (int64_t)e * H * I;
            for (int n = 0; n < H; ++n) {
                double acc = 0.0;
                for (int c = 0; c < I; ++c)
                    acc += (double)h[p * I + c] * (double)bf16_to_f32(We[(int64_t)n * I + c]);
                y[n] = static_cast<float>(acc);
            }
        }
    } else {
        if (H % 128 || I % 128) return 1;
        std::vector<uint8_t> qx(T * H), xq(R * H, 0), qh(R * I);
        std::vector<float> sx(T * (H / 128)), xs(R * (H / 128), 1.0f), sh(R * (I / 128));
        orc_quant_act_fp8(x, T, H, qx.data(), sx.data());
        orc_permute(qx.data(), sx.data(), 1, T, H, k, sorted_rows.data(), L, xq.data(), xs.data());
        orc_grouped_gemm_fp8(xq.data(), xs.data(), static_cast<const uint8_t*>(W1), W1s,
                             offsets.data(), E, R, 2 * I, H, nullptr, 0, Y1.data());
        orc_swiglu(Y1.data(), R, I, L, h.data());
        std::vector<uint16_t> hb(R * I);
        orc_bf16_round(h.data(), R * I, hb.data());
        orc_quant_act_fp8(hb.data(), R, I, qh.data(), sh.data());
        orc_grouped_gemm_fp8(qh.data(), sh.data(), static_cast<const uint8_t*>(W2), W2s,
                             offsets.data(), E, R, H, I, nullptr, 0, Y2.data());
    }
    orc_combine(Y2.data(), ids, w, row_pos.data(), T, k, H, E, out);
    if (sorted_rows_tap) std::copy(sorted_rows.begin(), sorted_rows.end(), sorted_rows_tap);
    if (row_pos_tap) std::copy(row_pos.begin(), row_pos.end(), row_pos_tap);
    if (offsets_tap) std::copy(offsets.begin(), offsets.end(), offsets_tap);
    return 0;
}

}  // extern "C"
