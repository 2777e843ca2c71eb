// Oracle for the fused fp16 GEMM  C = epilogue(A.B + bias).
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
// call this file; only the tests, the smoke check and the bench's CPU
// baseline use it.  It shares no code, header or table with the CUDA library.
//
// What it computes, for every checked output element (i, j):
//
//   acc = sum_{k=0..K-1} double(A[i,k]) * double(B[k,j])      (fp64, k ascending)
//   x   = acc + double(bias[j])          (bias is absent for the "none" epilogue)
//   y   = x                    epilogue none / bias
//         max(x, 0)            epilogue bias_relu
//         0.5 x (1 + erf(x/sqrt 2))   epilogue bias_gelu_erf
//         1 / (1 + exp(-x))    epilogue bias_sigmoid
//         0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))   epilogue bias_gelu_tanh
//   C[i,j] = fp16 round-to-nearest-even of y, straight from double.
//
// Sources, by page and section:
//   * "writing-tilelang-kernels", Kernel Anatomy and GEMM (Minimal): A is an
//     (M,K) fp16 tensor, B a (K,N) fp16 tensor, C an (M,N) fp16 tensor, the
//     accumulator is float; the PyTorch reference of the Step-by-Step
//     Workflow is the plain product A @ B.
//   * same page, Pre-flight Checklist pattern table: "GEMM + fusion" is a
//     ReLU (or sigmoid) epilogue after the GEMM.  The tanh form of GELU is
//     the common approximation of the exact one (the pages name GELU only).
//   * "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels from
//     Python", What you'll see and Why tile-level control matters: the fused
//     epilogue adds a bias and applies GELU while the accumulator is on chip,
//     then writes C once.  The GELU form is not given on the pages; the exact
//     erf form is the one this library implements.
//   * bias is a length-N vector broadcast over rows (Linear-layer reading;
//     the pages do not state its shape).
//
// The accumulation is done in fp64, i.e. more precisely than the fp32
// accumulator of the method, so the oracle is the mathematical definition
// rounded once; the GPU result differs from it by fp32 summation error plus
// one fp16 rounding, which the tests' tolerance covers.
//
// fp16 <-> double conversions are written here from the IEEE-754 binary16
// definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits,
// subnormals below 2^-14, Inf/NaN at exponent 31).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>
#include <algorithm>
#include <atomic>

namespace {

enum { EPI_NONE = 0, EPI_BIAS = 1, EPI_BIAS_RELU = 2, EPI_BIAS_GELU_ERF = 3, EPI_BIAS_SIGMOID = 4,
       EPI_BIAS_GELU_TANH = 5 };

double half_bits_to_double(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = std::ldexp(static_cast<double>(frac), -24);           // zero / subnormal
    } else if (expo == 31) {
        v = frac == 0 ? INFINITY : NAN;
    } else {
        v = std::ldexp(static_cast<double>(1024 + frac), expo - 25);  // (1.f) * 2^(e-15)
    }
    return sign ? -v : v;
}

// Round a non-negative double q (< 2^52) to the nearest integer, ties to even.
double round_half_even(double q) {
    const double fl = std::floor(q);
    const double diff = q - fl;  // exact: q and fl share the exponent range
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return std::fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

uint16_t double_to_half_bits(double x) {
    if (std::isnan(x)) return static_cast<uint16_t>(std::signbit(x) ? 0xfe00 : 0x7e00);
    const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
    const double a = std::fabs(x);
    // Largest finite fp16 is 65504; the midpoint to the next binade step
    // (65536) is 65520, which ties to the even neighbour 65536 = overflow.
    if (a >= 65520.0) return static_cast<uint16_t>(sign | 0x7c00);
    if (a < std::ldexp(1.0, -14)) {
        // Subnormal range: quantum 2^-24; a result of 1024 quanta is the
        // smallest normal, whose encoding is exactly 0x0400.
        const double q = round_half_even(std::ldexp(a, 24));
        return static_cast<uint16_t>(sign | static_cast<uint16_t>(q));
    }
    int e2 = 0;
    const double f = std::frexp(a, &e2);        // a = f * 2^e2, f in [0.5, 1)
    int expo = e2 - 1;                          // a in [2^expo, 2^(expo+1))
    double q = round_half_even(std::ldexp(f, 11));  // significand in [1024, 2048]
    if (q == 2048.0) { q = 1024.0; expo += 1; }
    if (expo > 15) return static_cast<uint16_t>(sign | 0x7c00);
    const int biased = expo + 15;
    return static_cast<uint16_t>(sign | (biased << 10) | (static_cast<int>(q) - 1024));
}

double apply_epilogue(double x, int epi) {
    switch (epi) {
        case EPI_BIAS_RELU:
            if (std::isnan(x)) return x;
            return x > 0.0 ? x : 0.0;
        case EPI_BIAS_GELU_ERF: return 0.5 * x * (1.0 + std::erf(x / std::sqrt(2.0)));
        case EPI_BIAS_SIGMOID: return 1.0 / (1.0 + std::exp(-x));
        case EPI_BIAS_GELU_TANH: {
            const double u = std::sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x);
            return 0.5 * x * (1.0 + std::tanh(u));
        }
        default: return x;
    }
}

std::vector<double> to_doubles(const uint16_t* p, int64_t n, int nthreads) {
    std::vector<double> out(static_cast<size_t>(n));
    const int64_t chunk = (n + nthreads - 1) / nthreads;
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) {
        const int64_t lo = t * chunk, hi = std::min<int64_t>(n, lo + chunk);
        if (lo >= hi) break;
        pool.emplace_back([=, &out] {
            for (int64_t i = lo; i < hi; ++i) out[static_cast<size_t>(i)] = half_bits_to_double(p[i]);
        });
    }
    for (auto& th : pool) th.join();
    return out;
}

int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    const unsigned hw = std::thread::hardware_concurrency();
    return hw ? static_cast<int>(hw) : 1;
}

bool bad_args(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
              int64_t M, int64_t N, int64_t K, int epi) {
    if (M < 0 || N < 0 || K < 0) return true;
    if (epi < EPI_NONE || epi > EPI_BIAS_GELU_TANH) return true;
    if (epi != EPI_NONE && bias == nullptr) return true;
    if (K > 0 && M > 0 && A == nullptr) return true;
    if (K > 0 && N > 0 && B == nullptr) return true;
    return false;
}

}  // namespace

extern "C" {

double oracle_half_to_double(uint16_t h) { return half_bits_to_double(h); }
uint16_t oracle_double_to_half(double x) { return double_to_half_bits(x); }
double oracle_epilogue(double x, int epi) { return apply_epilogue(x, epi); }

// Vector forms of the two conversions (used by the exhaustive pins).
void oracle_half_to_double_n(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = half_bits_to_double(h[i]);
}
void oracle_double_to_half_n(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = double_to_half_bits(x[i]);
}

// Full rows of C.  rows[r] selects the row of C written to out[r*N .. r*N+N).
// out_f64 (nullable) receives y before the fp16 rounding.  Returns 0 on
// success, 1 on bad arguments.
int oracle_gemm_rows(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                     int64_t M, int64_t N, int64_t K, int epi,
                     const int64_t* rows, int64_t nrows,
                     uint16_t* out, double* out_f64, int nthreads) {
    if (bad_args(A, B, bias, M, N, K, epi) || nrows < 0 || (nrows > 0 && !rows) || !out) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;
    nthreads = resolve_threads(nthreads);
    const std::vector<double> Bd = to_doubles(B, N * K, nthreads);
    std::vector<double> biasd(static_cast<size_t>(N), 0.0);
    if (epi != EPI_NONE)
        for (int64_t j = 0; j < N; ++j) biasd[static_cast<size_t>(j)] = half_bits_to_double(bias[j]);

    std::atomic<int64_t> next{0};
    auto worker = [&] {
        std::vector<double> acc(static_cast<size_t>(N));
        for (;;) {
            const int64_t r = next.fetch_add(1);
            if (r >= nrows) break;
            const int64_t i = rows[r];
            std::fill(acc.begin(), acc.end(), 0.0);
            for (int64_t k = 0; k < K; ++k) {
                const double a = half_bits_to_double(A[i * K + k]);
                const double* brow = Bd.data() + k * N;
                for (int64_t j = 0; j < N; ++j) acc[static_cast<size_t>(j)] += a * brow[j];
            }
            for (int64_t j = 0; j < N; ++j) {
                const double y = apply_epilogue(acc[static_cast<size_t>(j)] + biasd[static_cast<size_t>(j)], epi);
                out[r * N + j] = double_to_half_bits(y);
                if (out_f64) out_f64[r * N + j] = y;
            }
        }
    };
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
    return 0;
}

// Single elements (ii[e], jj[e]) of C, each a K-long fp64 dot product.
int oracle_gemm_elems(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                      int64_t M, int64_t N, int64_t K, int epi,
                      const int64_t* ii, const int64_t* jj, int64_t n,
                      uint16_t* out, double* out_f64, int nthreads) {
    if (bad_args(A, B, bias, M, N, K, epi) || n < 0 || (n > 0 && (!ii || !jj || !out))) return 1;
    for (int64_t e = 0; e < n; ++e)
        if (ii[e] < 0 || ii[e] >= M || jj[e] < 0 || jj[e] >= N) return 1;
    nthreads = resolve_threads(nthreads);
    std::atomic<int64_t> next{0};
    auto worker = [&] {
        for (;;) {
            const int64_t e = next.fetch_add(1);
            if (e >= n) break;
            const int64_t i = ii[e], j = jj[e];
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += half_bits_to_double(A[i * K + k]) * half_bits_to_double(B[k * N + j]);
            const double x = acc + (epi != EPI_NONE ? half_bits_to_double(bias[j]) : 0.0);
            const double y = apply_epilogue(x, epi);
            out[e] = double_to_half_bits(y);
            if (out_f64) out_f64[e] = y;
        }
    };
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
    return 0;
}

int oracle_default_threads(void) { return resolve_threads(0); }

}  // extern "C"
