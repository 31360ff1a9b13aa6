// W4A16 oracle: a plain, slow, obviously correct CPU statement of what the fused
// dequant-GEMM computes.  TEST INFRASTRUCTURE ONLY: nothing on the product path may
// include, link or call this file.  Only the tests, the smoke check and the bench's
// CPU-baseline leg load it (through oracle/__init__.py).  It shares no code, header,
// table or constant with the CUDA library in weight_only_int4_tma_gb300/.
//
// Sources (web pages, cited by title and section):
//   [P1] "W4A16 GEMM 算子浅析：INT4 权重反量化的计算流水线" (nxmr.cn)
//        - section "计算流水线的核心哲学": pipeline diagram, step 2
//          W_fp16 = (W_int4 - Zero) * Scale, then FP16 x FP16 -> FP32 MMA.
//        - section "Marlin 与 CUTLASS 中的寄存器解包黑魔法": one uint32 holds 8 nibbles.
//   [P3] "量化开销对比：各家方案的矩阵乘账本与省账手段" (laojiahuo2003.github.io)
//        - §3 route B: int4 -> unpack x scale -> FP16 -> FP16 GEMM.
//        - §6.2: the group scale lives on the reduction index k, so it is applied to the
//          weight operand; per-channel scales commute with the k-sum and go to the end.
//        - §6.4: group sizes 128 / 64 / 32.
//        - §6.7: per-channel scale folded into the epilogue.
//        - §6.2 (end of the tile pipeline: accumulator x scale -> + bias -> store) and
//          §6.6 (dequant + GEMM + scale + bias, + residual / activation, in one kernel):
//          the fused epilogue below.
//
// Readings where the pages are silent (each is listed in the design notes):
//   * nibble j of word w of a row is bits 4j..4j+3 and holds k = 8w + j (the pages
//     only say "8 per uint32");
//   * scales are dtype[K/g][N]; zeros are 4-bit, packed 8 per uint32 along N,
//     u32[K/g][N/8]; a missing zero array means every zero is 8 (symmetric);
//   * the dequantised weight is ONE round-to-nearest-even of the exact (q - z) * s into
//     the activation dtype; the k-sum is carried in fp64 here;
//   * the optional per-channel factor c[n] multiplies the finished fp64 sum.
//
// fp16 / bf16 encode and decode are written from the IEEE-754 definition below.
//
// Build: g++ -O2 -std=c++17 -fopenmp -shared -fPIC (see oracle/__init__.py).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---- IEEE-754 formats --------------------------------------------------------------
// binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.
// bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.
struct Fmt {
    int frac_bits;
    int exp_bits;
    int bias;
};
constexpr Fmt kF16{10, 5, 15};
constexpr Fmt kBF16{7, 8, 127};

inline const Fmt& fmt_of(int dtype) { return dtype == 0 ? kF16 : kBF16; }

// Decode: value = (-1)^s * 2^(e - bias) * (1 + f / 2^p) for 0 < e < max,
//         value = (-1)^s * 2^(1 - bias) * (f / 2^p)     for e == 0 (subnormal / zero).
double decode(uint16_t h, const Fmt& F) {
    const int p = F.frac_bits;
    const uint32_t emax_field = (1u << F.exp_bits) - 1u;
    const uint32_t s = h >> 15;
    const uint32_t e = (h >> p) & emax_field;
    const uint32_t f = h & ((1u << p) - 1u);
    double v;
    if (e == emax_field) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = std::ldexp(static_cast<double>(f), 1 - F.bias - p);
    } else {
        v = std::ldexp(static_cast<double>((1u << p) | f), static_cast<int>(e) - F.bias - p);
    }
    return s ? -v : v;
}

// Round an exact non-negative double n (n < 2^53) to an integer, ties to even.
double round_half_even(double n) {
    const double fl = std::floor(n);
    const double frac = n - fl;  // exact
    if (frac > 0.5) return fl + 1.0;
    if (frac < 0.5) return fl;
    return (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

// Encode: round-to-nearest-even of x into the format (overflow -> infinity).
uint16_t encode(double x, const Fmt& F) {
    const int p = F.frac_bits;
    const uint32_t emax_field = (1u << F.exp_bits) - 1u;
    const int emin = 1 - F.bias;               // smallest normal exponent
    const int emax = static_cast<int>(emax_field) - 1 - F.bias;  // largest normal exponent
    if (std::isnan(x)) return static_cast<uint16_t>((emax_field << p) | (1u << (p - 1)));
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    const double a = std::fabs(x);
    if (std::isinf(a)) return static_cast<uint16_t>(sign | (emax_field << p));
    if (a == 0.0) return sign;
    int E;
    (void)std::frexp(a, &E);                   // a = m * 2^E, m in [0.5, 1)
    int e = E - 1;                             // a in [2^e, 2^(e+1))
    if (e < emin) e = emin;                    // subnormal range shares the emin quantum
    // Quantum (spacing of representable values) at this exponent.
    const double n = std::ldexp(a, p - e);     // a / 2^(e - p), exact
    const double r = round_half_even(n);       // integer in [0, 2^(p+1)]
    // Rounded magnitude is r * 2^(e - p).
    if (r >= std::ldexp(1.0, p + 1)) {         // carried into the next binade
        const int e2 = e + 1;
        if (e2 > emax) return static_cast<uint16_t>(sign | (emax_field << p));
        return static_cast<uint16_t>(sign | (static_cast<uint32_t>(e2 + F.bias) << p));
    }
    const uint32_t ri = static_cast<uint32_t>(r);
    if (ri < (1u << p)) {                      // subnormal (only possible when e == emin)
        return static_cast<uint16_t>(sign | ri);
    }
    if (e > emax) return static_cast<uint16_t>(sign | (emax_field << p));
    return static_cast<uint16_t>(sign | (static_cast<uint32_t>(e + F.bias) << p) |
                                 (ri & ((1u << p) - 1u)));
}

// Spacing of representable values at |v| (the unit in the last place of v's binade).
double ulp_of(uint16_t h, const Fmt& F) {
    const int p = F.frac_bits;
    const uint32_t emax_field = (1u << F.exp_bits) - 1u;
    const uint32_t e = (h >> p) & emax_field;
    if (e == emax_field) return INFINITY;
    const int ee = (e == 0) ? 1 : static_cast<int>(e);
    return std::ldexp(1.0, ee - F.bias - p);
}

// ---- unpack [P1 "寄存器解包黑魔法": 8 nibbles per uint32] -----------------------------
inline int nibble_q(const uint32_t* qweight, int K, int n, int k) {
    const uint32_t w = qweight[static_cast<size_t>(n) * (K / 8) + k / 8];
    return static_cast<int>((w >> (4 * (k % 8))) & 0xFu);
}

inline int nibble_z(const uint32_t* qzeros, int N, int gi, int n) {
    if (qzeros == nullptr) return 8;  // symmetric: zero fixed at 8
    const uint32_t w = qzeros[static_cast<size_t>(gi) * (N / 8) + n / 8];
    return static_cast<int>((w >> (4 * (n % 8))) & 0xFu);
}

// ---- dequant [P1 "计算流水线的核心哲学" step 2; P3 §6.2] -------------------------------
// Wd[n,k] = RNE_dtype( (q[n,k] - z[k/g, n]) * s[k/g, n] ).  The product of an integer in
// [-15, 15] and an 11-bit (or 8-bit) significand is exact in fp64, so the only rounding
// is the final encode.
inline uint16_t dequant_one(const uint32_t* qweight, const uint16_t* scales,
                            const uint32_t* qzeros, int N, int K, int group, const Fmt& F,
                            int n, int k) {
    const int gi = k / group;
    const int q = nibble_q(qweight, K, n, k);
    const int z = nibble_z(qzeros, N, gi, n);
    const double s = decode(scales[static_cast<size_t>(gi) * N + n], F);
    return encode(static_cast<double>(q - z) * s, F);
}

bool shape_ok(int N, int K, int group) {
    return N > 0 && K > 0 && group > 0 && K % group == 0 && K % 8 == 0 && N % 8 == 0;
}

}  // namespace

extern "C" {

int w4o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double w4o_decode(uint16_t h, int dtype) { return decode(h, fmt_of(dtype)); }
uint16_t w4o_encode(double x, int dtype) { return encode(x, fmt_of(dtype)); }
double w4o_ulp(uint16_t h, int dtype) { return ulp_of(h, fmt_of(dtype)); }

void w4o_decode_array(const uint16_t* h, int64_t count, int dtype, double* out) {
    const Fmt& F = fmt_of(dtype);
    for (int64_t i = 0; i < count; ++i) out[i] = decode(h[i], F);
}

void w4o_encode_array(const double* x, int64_t count, int dtype, uint16_t* out) {
    const Fmt& F = fmt_of(dtype);
    for (int64_t i = 0; i < count; ++i) out[i] = encode(x[i], F);
}

// q[n*K + k] = nibble k of row n.
int w4o_unpack_q(const uint32_t* qweight, int N, int K, uint8_t* q) {
    if (K % 8 != 0 || N <= 0 || K <= 0) return -1;
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            q[static_cast<size_t>(n) * K + k] = static_cast<uint8_t>(nibble_q(qweight, K, n, k));
    return 0;
}

// z[gi*N + n] = zero of group gi, column n (8 everywhere when qzeros is NULL).
int w4o_unpack_z(const uint32_t* qzeros, int G, int N, uint8_t* z) {
    if (N % 8 != 0 || N <= 0 || G <= 0) return -1;
    for (int gi = 0; gi < G; ++gi)
        for (int n = 0; n < N; ++n)
            z[static_cast<size_t>(gi) * N + n] = static_cast<uint8_t>(nibble_z(qzeros, N, gi, n));
    return 0;
}

// Wd[n*K + k] = dtype bits of the dequantised weight.
int w4o_dequant(const uint32_t* qweight, const uint16_t* scales, const uint32_t* qzeros,
                int N, int K, int group, int dtype, uint16_t* Wd) {
    if (!shape_ok(N, K, group)) return -1;
    const Fmt& F = fmt_of(dtype);
#pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k)
            Wd[static_cast<size_t>(n) * K + k] =
                dequant_one(qweight, scales, qzeros, N, K, group, F, n, k);
    return 0;
}

// Full product from already-dequantised weights.
//   Yd[m,n]   = c[n] * sum_k A[m,k] * Wd[n,k]      (fp64, k ascending)
//   Babs[m,n] = |c[n]| * sum_k |A[m,k] * Wd[n,k]|
//   Yref[m,n] = RNE_dtype(Yd[m,n])
// cscale (dtype bits [N]) may be NULL (c = 1).  Any output pointer may be NULL.
int w4o_gemm(const uint16_t* A, const uint16_t* Wd, const uint16_t* cscale, int M, int N,
             int K, int dtype, double* Yd, double* Babs, uint16_t* Yref) {
    if (M <= 0 || N <= 0 || K <= 0) return -1;
    const Fmt& F = fmt_of(dtype);
    std::vector<double> Ad(static_cast<size_t>(M) * K);
    for (size_t i = 0; i < Ad.size(); ++i) Ad[i] = decode(A[i], F);
#pragma omp parallel
    {
        std::vector<double> w(K);
#pragma omp for schedule(dynamic, 4)
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) w[k] = decode(Wd[static_cast<size_t>(n) * K + k], F);
            const double c = cscale ? decode(cscale[n], F) : 1.0;
            for (int m = 0; m < M; ++m) {
                const double* a = &Ad[static_cast<size_t>(m) * K];
                double acc = 0.0, mag = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double t = a[k] * w[k];
                    acc += t;
                    mag += std::fabs(t);
                }
                const size_t o = static_cast<size_t>(m) * N + n;
                const double y = c * acc;
                if (Yd) Yd[o] = y;
                if (Babs) Babs[o] = std::fabs(c) * mag;
                if (Yref) Yref[o] = encode(y, F);
            }
        }
    }
    return 0;
}

// The same quantities for a list of (m, n) positions, dequantising on the fly from the
// canonical (q, s, z) inputs.  Used at sizes where the full product is too slow.
int w4o_gemm_sampled(const uint16_t* A, const uint32_t* qweight, const uint16_t* scales,
                     const uint32_t* qzeros, const uint16_t* cscale, int M, int N, int K,
                     int group, int dtype, const int64_t* idx_m, const int64_t* idx_n,
                     int64_t count, double* Yd, double* Babs, uint16_t* Yref) {
    if (!shape_ok(N, K, group) || M <= 0) return -1;
    const Fmt& F = fmt_of(dtype);
    for (int64_t i = 0; i < count; ++i)
        if (idx_m[i] < 0 || idx_m[i] >= M || idx_n[i] < 0 || idx_n[i] >= N) return -2;
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < count; ++i) {
        const int m = static_cast<int>(idx_m[i]);
        const int n = static_cast<int>(idx_n[i]);
        double acc = 0.0, mag = 0.0;
        for (int k = 0; k < K; ++k) {
            const double w = decode(dequant_one(qweight, scales, qzeros, N, K, group, F, n, k), F);
            const double t = decode(A[static_cast<size_t>(m) * K + k], F) * w;
            acc += t;
            mag += std::fabs(t);
        }
        const double c = cscale ? decode(cscale[n], F) : 1.0;
        const double y = c * acc;
        if (Yd) Yd[i] = y;
        if (Babs) Babs[i] = std::fabs(c) * mag;
        if (Yref) Yref[i] = encode(y, F);
    }
    return 0;
}

// The product with weights that are NOT rounded to the activation dtype: the integer-
// operand variant (the MMA takes the exact q - z, the group scale multiplies each group's
// partial sum: "fine-grained" per-group scaling; [P3] §6.2 explains why the group scale
// cannot move past the whole k-sum, only past each group's part of it).  Mathematically the k-sum of
//   A[m,k] * (q[n,k] - z[k/g,n]) * s[k/g,n]
// with every term exact in fp64 (no encode of the weight):
//   Yd[m,n] = c[n] * sum_k A[m,k] (q - z) s,   Babs[m,n] = |c[n]| * sum_k |A[m,k] (q - z) s|.
int w4o_gemm_exact_w(const uint16_t* A, const uint32_t* qweight, const uint16_t* scales,
                     const uint32_t* qzeros, const uint16_t* cscale, int M, int N, int K,
                     int group, int dtype, double* Yd, double* Babs, uint16_t* Yref) {
    if (!shape_ok(N, K, group) || M <= 0) return -1;
    const Fmt& F = fmt_of(dtype);
    std::vector<double> Ad(static_cast<size_t>(M) * K);
    for (size_t i = 0; i < Ad.size(); ++i) Ad[i] = decode(A[i], F);
#pragma omp parallel
    {
        std::vector<double> w(K);
#pragma omp for schedule(dynamic, 4)
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) {
                const int gi = k / group;
                const int q = nibble_q(qweight, K, n, k);
                const int z = nibble_z(qzeros, N, gi, n);
                w[k] = static_cast<double>(q - z) * decode(scales[static_cast<size_t>(gi) * N + n], F);
            }
            const double c = cscale ? decode(cscale[n], F) : 1.0;
            for (int m = 0; m < M; ++m) {
                const double* a = &Ad[static_cast<size_t>(m) * K];
                double acc = 0.0, mag = 0.0;
                for (int k = 0; k < K; ++k) {
                    const double t = a[k] * w[k];
                    acc += t;
                    mag += std::fabs(t);
                }
                const size_t o = static_cast<size_t>(m) * N + n;
                const double y = c * acc;
                if (Yd) Yd[o] = y;
                if (Babs) Babs[o] = std::fabs(c) * mag;
                if (Yref) Yref[o] = encode(y, F);
            }
        }
    }
    return 0;
}

// Element-wise acceptance test:  |Y - Yd| <= rel_tol * Babs + ulp_dtype(RNE_dtype(Yd)).
// Returns the number of failing elements; *first_bad receives the first failing index
// (or -1) and *worst the largest |Y - Yd| / (rel_tol * Babs + ulp) seen.
int64_t w4o_check(const uint16_t* Y, const double* Yd, const double* Babs, int64_t count,
                  int dtype, double rel_tol, int64_t* first_bad, double* worst) {
    const Fmt& F = fmt_of(dtype);
    int64_t bad = 0, first = -1;
    double wr = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        const double y = decode(Y[i], F);
        const double bound = rel_tol * Babs[i] + ulp_of(encode(Yd[i], F), F);
        const double err = std::fabs(y - Yd[i]);
        const double ratio = (bound > 0.0) ? err / bound : (err == 0.0 ? 0.0 : INFINITY);
        if (!(err <= bound)) {  // NaN fails too
            if (first < 0) first = i;
            ++bad;
        }
        if (!(ratio <= wr)) wr = ratio;
    }
    if (first_bad) *first_bad = first;
    if (worst) *worst = wr;
    return bad;
}

// Fused epilogue ("量化开销对比" §6.2, §6.6).  From the GEMM's fp64 result Yd (per-channel
// factor included) and its magnitude Babs, per element (m, n):
//     pre  = Yd + bias[n]                      (bias optional)
//     post = act(pre)                          0: identity, 1: max(pre, 0),
//                                              2: SiLU, pre / (1 + exp(-pre))
//     out  = post + residual[m, n]             (residual optional)
// all in fp64 (the pages fix no order between residual and activation; the activation
// is applied to the biased GEMM result and the residual added after it).  Also
//     Bout = L * Babs + |bias| + |residual|     L = 1 (identity, ReLU) or 1.1 (SiLU,
//                                               whose slope lies in [-0.1, 1.1])
// the magnitude that scales the fused result's error bound, and Yref = RNE_dtype(out).
int w4o_epilogue(const double* Yd, const double* Babs, const uint16_t* bias,
                 const uint16_t* residual, int act, int M, int N, int dtype, double* Yout,
                 double* Bout, uint16_t* Yref) {
    if (M <= 0 || N <= 0 || act < 0 || act > 2) return -1;
    const Fmt& F = fmt_of(dtype);
    const double L = act == 2 ? 1.1 : 1.0;
    for (int m = 0; m < M; ++m) {
        for (int n = 0; n < N; ++n) {
            const size_t o = static_cast<size_t>(m) * N + n;
            const double b = bias ? decode(bias[n], F) : 0.0;
            const double r = residual ? decode(residual[o], F) : 0.0;
            const double pre = Yd[o] + b;
            double post = pre;
            if (act == 1) post = pre > 0.0 ? pre : 0.0;
            if (act == 2) post = pre / (1.0 + std::exp(-pre));
            const double out = post + r;
            if (Yout) Yout[o] = out;
            if (Bout) Bout[o] = L * Babs[o] + std::fabs(b) + std::fabs(r);
            if (Yref) Yref[o] = encode(out, F);
        }
    }
    return 0;
}

}  // extern "C"
