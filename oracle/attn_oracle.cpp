// Oracle for attention forward:  O = softmax(scale * Q K^T) V  per (batch, head).
//
// TEST INFRASTRUCTURE ONLY, like gemm_oracle.cpp (whose IEEE binary16
// conversions it calls): only the tests and the bench's CPU legs use it.  It
// shares no code with the CUDA library.
//
// For every requested query row i of head (b, h):
//
//   s_j  = scale * sum_{d=0..D-1} double(Q[b,h,i,d]) * double(K[b,h,j,d])   for j in A(i)
//   p_j  = exp(s_j - max_{j' in A(i)} s_j') / sum_{j' in A(i)} exp(s_j' - max)
//   O[b,h,i,d] = fp16_rne( sum_{j in A(i)} p_j * double(V[b,h,j,d]) )
//
// with A(i) = {0 .. S-1} (non-causal) or {0 .. i} (causal), all in double,
// rounded once.  Q, K, V, O are (B, H, S, D) row-major fp16.
//
// Sources, by page and section:
//   * "writing-tilelang-kernels", Flash Attention Forward: the kernel's
//     signature, Q, K, V and O as (B, H, S, D) float16 tensors; the pattern
//     table's "Online Softmax" (running max, exp, rescaling) and "Flash
//     Attention" rows.
//   * "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels from
//     Python", FlashAttention: the FLOP model and what the example measures:
//     softmax computed online without materialising the S x S matrix, causal
//     and non-causal, validated against torch's scaled_dot_product_attention.
//     The pages give no scale; SDPA's default 1/sqrt(D) is the plain reading
//     (the caller passes the scale), and SDPA's causal mask keeps key j for
//     query i when j <= i.
//
// Subtracting the row maximum does not change p (it cancels in the ratio);
// it keeps exp() in range.  The oracle is the definition, evaluated directly:
// there is no online rescaling here.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

extern "C" double oracle_half_to_double(uint16_t h);
extern "C" uint16_t oracle_double_to_half(double x);

extern "C" {

// Rows rows[r] = (b * H + h) * S + i of O, written to out[r * D .. r * D + D).
// out_f64 (nullable) receives the values before rounding.  Returns 0 on
// success, 1 on bad arguments.
int oracle_attn_rows(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B, int64_t H, int64_t S,
                     int64_t D, int causal, double scale, const int64_t* rows, int64_t nrows, uint16_t* out,
                     double* out_f64, int nthreads) {
    if (B < 0 || H < 0 || S < 0 || D <= 0 || nrows < 0) return 1;
    if (nrows > 0 && (!Q || !K || !V || !rows || !out)) return 1;
    const int64_t total = B * H * S;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return 1;
    if (nthreads <= 0) {
        const unsigned hw = std::thread::hardware_concurrency();
        nthreads = hw ? static_cast<int>(hw) : 1;
    }
    std::atomic<int64_t> next{0};
    auto worker = [&] {
        std::vector<double> q(static_cast<size_t>(D)), s(static_cast<size_t>(S)), o(static_cast<size_t>(D));
        for (;;) {
            const int64_t r = next.fetch_add(1);
            if (r >= nrows) break;
            const int64_t row = rows[r];
            const int64_t bh = row / S, i = row - bh * S;
            const uint16_t* Qh = Q + bh * S * D;
            const uint16_t* Kh = K + bh * S * D;
            const uint16_t* Vh = V + bh * S * D;
            const int64_t nkeys = causal ? i + 1 : S;
            for (int64_t d = 0; d < D; ++d) q[static_cast<size_t>(d)] = oracle_half_to_double(Qh[i * D + d]);
            double mx = -INFINITY;
            for (int64_t j = 0; j < nkeys; ++j) {
                double acc = 0.0;
                for (int64_t d = 0; d < D; ++d) acc += q[static_cast<size_t>(d)] * oracle_half_to_double(Kh[j * D + d]);
                s[static_cast<size_t>(j)] = scale * acc;
                mx = std::max(mx, s[static_cast<size_t>(j)]);
            }
            double denom = 0.0;
            for (int64_t j = 0; j < nkeys; ++j) {
                s[static_cast<size_t>(j)] = std::exp(s[static_cast<size_t>(j)] - mx);
                denom += s[static_cast<size_t>(j)];
            }
            std::fill(o.begin(), o.end(), 0.0);
            for (int64_t j = 0; j < nkeys; ++j) {
                const double p = s[static_cast<size_t>(j)] / denom;
                for (int64_t d = 0; d < D; ++d) o[static_cast<size_t>(d)] += p * oracle_half_to_double(Vh[j * D + d]);
            }
            for (int64_t d = 0; d < D; ++d) {
                out[r * D + d] = oracle_double_to_half(o[static_cast<size_t>(d)]);
                if (out_f64) out_f64[r * D + d] = o[static_cast<size_t>(d)];
            }
        }
    };
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
    return 0;
}

}  // extern "C"
