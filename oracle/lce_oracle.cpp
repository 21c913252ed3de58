// Plain fp64 C++ oracle for the fused output-projection + cross-entropy path.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path links or calls this
// file: only the tests, the package's smoke check and the benchmark's CPU
// baseline load it (through ctypes, as oracle/liblce_oracle.so). It shares no
// code, header or constant with the CUDA library.
//
// It computes the plain definition in double precision on the exact input
// values (float64, float32 or bf16 bit patterns, each widened exactly):
//
//   valid rows    I = { i : t_i != ignore_index }, ascending, Nv = |I|
//   logits        s_iv = sum_k H[i,k] W[v,k]
//   log-sum-exp   lse_i = M_i + log sum_v exp(s_iv - M_i),  M_i = max_v s_iv
//   loss          loss = (1/Nv) sum_{i in I} (lse_i - s_{i,t_i})
//   softmax grad  g_iv = (exp(s_iv - lse_i) - [v == t_i]) / Nv
//   dH[i,:]       = sum_v g_iv W[v,:]  for i in I, zero on ignored rows
//   dW[v,:]       = sum_{i in I} g_iv H[i,:]
//
// Sources: the projection plus loss streamed in chunks with padding tokens
// skipped ("OjasX 0.6.1: Training a 1B-Parameter LLM in 6.35GB of RAM",
// section "Core Technology", the zero-byte vocabulary logits item); logits
// recomputed in backward instead of stored, which leaves the gradients as they
// are ("6GB显卡预训练11亿参数模型", sections "内存实际花在哪里" and "关键参数说明",
// --chunked-loss 512); the online softmax reaching the same result as the
// two-pass one (same OjasX page, "Online Softmax" note). The normaliser is the
// number of valid tokens; Nv = 0 gives a NaN loss and zero gradients (the
// mean over an empty set). A target outside [0, V) that is not ignore_index is
// an input error: the call returns LCEO_ERR_TARGET and writes nothing.
//
// Structure: one pass over the valid rows (a row at a time: its V logits, the
// whole-row max and log-sum-exp, its loss and its dH row), then one pass over
// the vocabulary rows (a row v at a time: dW[v,:] as the sum over valid i in
// ascending order, each s_iv recomputed from H and W). Each row's max and
// log-sum-exp are taken over the complete row, never by a streaming
// recurrence. std::thread splits the rows of each pass; every output element
// is produced by one thread in a fixed order and the loss is summed in
// ascending row order afterwards, so the results do not depend on the thread
// count. The one liberty taken with rounding order: a dot product over k is
// accumulated in eight interleaved partial sums (k mod 8) added pairwise at
// the end, so that the compiler can keep several additions in flight.
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

enum : int { LCEO_OK = 0, LCEO_ERR_ARG = 1, LCEO_ERR_TARGET = 2 };
enum : int { IN_F64 = 0, IN_F32 = 1, IN_BF16 = 2 };

inline double widen(double x) { return x; }
inline double widen(float x) { return static_cast<double>(x); }
// bf16 bit pattern -> its exact value (the top 16 bits of an fp32)
inline double widen(uint16_t b) {
    const uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

// One row of an input matrix widened to double.
template <typename T>
void widen_row(const T *src, int64_t d, double *dst) {
    for (int64_t k = 0; k < d; ++k) dst[k] = widen(src[k]);
}

template <typename T>
double dot(const double *a, const T *b, int64_t d) {
    double p[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int64_t k = 0;
    for (; k + 8 <= d; k += 8)
        for (int j = 0; j < 8; ++j) p[j] += a[k + j] * widen(b[k + j]);
    for (int j = 0; k < d; ++k, ++j) p[j] += a[k] * widen(b[k]);
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// acc += g * x (x widened element by element)
template <typename T>
void axpy(double g, const T *x, int64_t d, double *acc) {
    for (int64_t k = 0; k < d; ++k) acc[k] += g * widen(x[k]);
}

// Run f(lo, hi) over [0, n) split into `threads` contiguous ranges.
template <typename F>
void parallel_for(int64_t n, int threads, F f) {
    if (threads < 1) threads = 1;
    if (n < threads) threads = static_cast<int>(n > 0 ? n : 1);
    if (threads == 1) {
        f(int64_t{0}, n);
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 0; t < threads; ++t) {
        const int64_t lo = n * t / threads, hi = n * (t + 1) / threads;
        pool.emplace_back([=] { f(lo, hi); });
    }
    for (auto &th : pool) th.join();
}

struct Problem {
    const void *H, *W;
    int dtype;
    const int64_t *t;
    int64_t ignore, N, d, V;
    int threads;
};

// Pass over valid rows: lse_i, the loss term and (when wanted) dH row i.
// rows: the valid rows to process (ascending positions); nv: the normaliser.
template <typename T>
void row_pass(const Problem &p, const std::vector<int64_t> &rows, int64_t nv, double *lse_out,
              double *loss_rows, double *dH_rows /* [rows.size()][d] or null */) {
    const T *H = static_cast<const T *>(p.H);
    const T *W = static_cast<const T *>(p.W);
    const int64_t d = p.d, V = p.V;
    parallel_for(static_cast<int64_t>(rows.size()), p.threads, [&](int64_t lo, int64_t hi) {
        std::vector<double> h(d), s(V), acc(d);
        for (int64_t j = lo; j < hi; ++j) {
            const int64_t i = rows[j];
            widen_row(H + i * d, d, h.data());
            for (int64_t v = 0; v < V; ++v) s[v] = dot(h.data(), W + v * d, d);   // s_iv for all v
            double M = -std::numeric_limits<double>::infinity();   // M_i = max_v s_iv
            for (int64_t v = 0; v < V; ++v) M = s[v] > M ? s[v] : M;
            double sum = 0.0;                                       // sum_v exp(s_iv - M_i)
            for (int64_t v = 0; v < V; ++v) sum += std::exp(s[v] - M);
            const double lse = M + std::log(sum);
            const int64_t ti = p.t[i];
            lse_out[j] = lse;
            loss_rows[j] = lse - s[ti];
            if (dH_rows) {                                          // dH_i = sum_v g_iv W_v
                std::fill(acc.begin(), acc.end(), 0.0);
                for (int64_t v = 0; v < V; ++v) {
                    const double g = (std::exp(s[v] - lse) - (v == ti ? 1.0 : 0.0)) / static_cast<double>(nv);
                    axpy(g, W + v * d, d, acc.data());
                }
                std::memcpy(dH_rows + j * d, acc.data(), sizeof(double) * d);
            }
        }
    });
}

// Pass over vocabulary rows: dW[v,:] = sum over valid i (ascending) of g_iv H_i,
// with s_iv recomputed and lse_i taken from the row pass.
template <typename T>
void vocab_pass(const Problem &p, const std::vector<int64_t> &valid, const double *lse_valid, int64_t nv,
                const std::vector<int64_t> &vocab, double *dW_rows /* [vocab.size()][d] */) {
    const T *H = static_cast<const T *>(p.H);
    const T *W = static_cast<const T *>(p.W);
    const int64_t d = p.d;
    parallel_for(static_cast<int64_t>(vocab.size()), p.threads, [&](int64_t lo, int64_t hi) {
        std::vector<double> w(d), acc(d);
        for (int64_t j = lo; j < hi; ++j) {
            const int64_t v = vocab[j];
            widen_row(W + v * d, d, w.data());
            std::fill(acc.begin(), acc.end(), 0.0);
            for (size_t q = 0; q < valid.size(); ++q) {
                const int64_t i = valid[q];
                const double s = dot(w.data(), H + i * d, d);
                const double g = (std::exp(s - lse_valid[q]) - (p.t[i] == v ? 1.0 : 0.0)) / static_cast<double>(nv);
                axpy(g, H + i * d, d, acc.data());
            }
            std::memcpy(dW_rows + j * d, acc.data(), sizeof(double) * d);
        }
    });
}

int check(const Problem &p, std::vector<int64_t> &valid) {
    if (!p.H || !p.W || !p.t || p.N < 0 || p.d < 1 || p.V < 1) return LCEO_ERR_ARG;
    if (p.dtype != IN_F64 && p.dtype != IN_F32 && p.dtype != IN_BF16) return LCEO_ERR_ARG;
    valid.clear();
    for (int64_t i = 0; i < p.N; ++i) {
        const int64_t ti = p.t[i];
        if (ti == p.ignore) continue;
        if (ti < 0 || ti >= p.V) return LCEO_ERR_TARGET;
        valid.push_back(i);
    }
    return LCEO_OK;
}

template <typename F>
void by_dtype(int dtype, F f) {
    if (dtype == IN_F64)
        f(double{});
    else if (dtype == IN_F32)
        f(float{});
    else
        f(uint16_t{});
}

double mean_loss(const std::vector<double> &loss_rows) {
    if (loss_rows.empty()) return std::numeric_limits<double>::quiet_NaN();
    double sum = 0.0;
    for (double x : loss_rows) sum += x;   // ascending row order
    return sum / static_cast<double>(loss_rows.size());
}

}  // namespace

extern "C" {

// Valid-row count and positions (ascending) of targets != ignore_index.
// With V > 0, returns LCEO_ERR_TARGET if a non-ignored target lies outside
// [0, V); with V <= 0 the targets are not range-checked.
int lceo_valid_rows(const int64_t *t, int64_t ignore, int64_t N, int64_t V, int64_t *idx_out, int64_t *nv_out) {
    if (!t || !nv_out || N < 0) return LCEO_ERR_ARG;
    int64_t nv = 0;
    for (int64_t i = 0; i < N; ++i) {
        if (t[i] == ignore) continue;
        if (V > 0 && (t[i] < 0 || t[i] >= V)) return LCEO_ERR_TARGET;
        if (idx_out) idx_out[nv] = i;
        ++nv;
    }
    *nv_out = nv;
    return LCEO_OK;
}

// Loss, per-position lse (NaN at ignored positions) and loss terms; dH [N][d]
// and dW [V][d] when non-null. Inputs: H [N][d], W [V][d] of `dtype`
// (0 float64, 1 float32, 2 bf16 bits), t [N] int64.
int lceo_forward_backward(const void *H, const void *W, int dtype, const int64_t *t, int64_t ignore, int64_t N,
                          int64_t d, int64_t V, int threads, double *loss, double *lse, double *loss_terms,
                          double *dH, double *dW) {
    Problem p{H, W, dtype, t, ignore, N, d, V, threads};
    std::vector<int64_t> valid;
    const int rc = check(p, valid);
    if (rc || !loss) return rc ? rc : LCEO_ERR_ARG;
    const int64_t nv = static_cast<int64_t>(valid.size());
    std::vector<double> lse_v(nv), loss_v(nv), dH_v(dH ? nv * d : 0);
    by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        row_pass<T>(p, valid, nv, lse_v.data(), loss_v.data(), dH ? dH_v.data() : nullptr);
        if (dW) {
            std::vector<int64_t> all(V);
            for (int64_t v = 0; v < V; ++v) all[v] = v;
            vocab_pass<T>(p, valid, lse_v.data(), nv, all, dW);
        }
    });
    *loss = mean_loss(loss_v);
    const double nan = std::numeric_limits<double>::quiet_NaN();
    if (lse) for (int64_t i = 0; i < N; ++i) lse[i] = nan;
    if (loss_terms) for (int64_t i = 0; i < N; ++i) loss_terms[i] = nan;
    if (dH) std::memset(dH, 0, sizeof(double) * N * d);
    for (int64_t q = 0; q < nv; ++q) {
        const int64_t i = valid[q];
        if (lse) lse[i] = lse_v[q];
        if (loss_terms) loss_terms[i] = loss_v[q];
        if (dH) std::memcpy(dH + i * d, dH_v.data() + q * d, sizeof(double) * d);
    }
    return LCEO_OK;
}

// For shapes too large for the full gradients: the loss and every valid
// position's lse (as lceo_forward_backward), dH on `n_rows` positions
// (zero rows where ignored) and dW on `n_vocab` vocabulary rows. dW[v] needs
// g_iv for every valid i, hence every valid row's lse; dH[i] needs row i's
// logits only.
int lceo_sampled(const void *H, const void *W, int dtype, const int64_t *t, int64_t ignore, int64_t N, int64_t d,
                 int64_t V, int threads, const int64_t *rows, int64_t n_rows, const int64_t *vocab, int64_t n_vocab,
                 double *loss, double *lse, double *dH_rows, double *dW_rows) {
    Problem p{H, W, dtype, t, ignore, N, d, V, threads};
    std::vector<int64_t> valid;
    const int rc = check(p, valid);
    if (rc || !loss || (n_rows && (!rows || !dH_rows)) || (n_vocab && (!vocab || !dW_rows))) return rc ? rc : LCEO_ERR_ARG;
    for (int64_t j = 0; j < n_rows; ++j)
        if (rows[j] < 0 || rows[j] >= N) return LCEO_ERR_ARG;
    for (int64_t j = 0; j < n_vocab; ++j)
        if (vocab[j] < 0 || vocab[j] >= V) return LCEO_ERR_ARG;
    const int64_t nv = static_cast<int64_t>(valid.size());
    std::vector<double> lse_v(nv), loss_v(nv);
    std::vector<int64_t> sel;          // sampled positions that are valid
    std::vector<int64_t> sel_at;       // their slot in `rows`
    for (int64_t j = 0; j < n_rows; ++j)
        if (t[rows[j]] != ignore) {
            sel.push_back(rows[j]);
            sel_at.push_back(j);
        }
    std::vector<double> sel_lse(sel.size()), sel_loss(sel.size()), sel_dH(sel.size() * d);
    by_dtype(dtype, [&](auto tag) {
        using T = decltype(tag);
        row_pass<T>(p, valid, nv, lse_v.data(), loss_v.data(), nullptr);
        if (!sel.empty()) row_pass<T>(p, sel, nv, sel_lse.data(), sel_loss.data(), sel_dH.data());
        if (n_vocab) {
            std::vector<int64_t> vv(vocab, vocab + n_vocab);
            vocab_pass<T>(p, valid, lse_v.data(), nv, vv, dW_rows);
        }
    });
    *loss = mean_loss(loss_v);
    if (lse) {
        for (int64_t i = 0; i < N; ++i) lse[i] = std::numeric_limits<double>::quiet_NaN();
        for (int64_t q = 0; q < nv; ++q) lse[valid[q]] = lse_v[q];
    }
    if (n_rows) std::memset(dH_rows, 0, sizeof(double) * n_rows * d);
    for (size_t q = 0; q < sel.size(); ++q)
        std::memcpy(dH_rows + sel_at[q] * d, sel_dH.data() + q * d, sizeof(double) * d);
    return LCEO_OK;
}

}  // extern "C"
