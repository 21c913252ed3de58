// Host runtime and C ABI of liblce: argument checks, workspace layout, TMA
// tensor-map encoding, and the launch sequence of the fused output-projection
// + cross-entropy path on the caller's stream.
//
// Sequence (all on `stream`, no host synchronisation), per token chunk
// (all N rows unless lce_args_t.token_chunk caps it; k_count_valid first
// counts the call's valid rows when there are several chunks):
//   1 k_compact        valid rows -> idx / inv / Nv (device)
//   2 k_gather         Hc = H[idx], zero-padded to 256-row pair blocks (with
//                      row_gather: no copy, the GEMMs gather H's rows by
//                      TMA gather4; only targets and the padded index
//                      entries are written)
//   3 k_gemm<LSE>      logits tiles + online log-sum-exp partials + target logit
//   4 k_lse_merge      lse per row, loss_i
//   5 k_loss_partial   sum of loss_i (k_loss_final: loss = sum / Nv)
//   backward, one launch per vocab chunk j of Vc rows (j = -1 .. chunks-1):
//   6 k_gemm<BWD>      G_{j+1} = (softmax - onehot)/Nv from recomputed logits
//                      of chunk j+1, dW[chunk j] = G_j^T Hc and
//                      dHacc (+)= G_j W[chunk j] (three G buffers; consecutive
//                      launches overlap through programmatic dependent launch;
//                      with a fused optimizer, k_gemm<BWD_OPT>: dW tiles of
//                      chunk j one launch later, applying SGD / AdamW to W,
//                      four G buffers, launches j = -1 .. chunks)
//   7 k_dh_scatter     dH = dHacc[inv], zero on ignored rows
// and finally k_loss_final (loss = sum of the chunks' sums / Nv). With a
// stored lse (lse_in), k_lse_from_input replaces steps 3-5.
// The input-embedding lookup and its gradient (lce_embedding_*) are separate
// entry points over the kernels of lce_embed.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "lce.h"
#include "lce_embed.cuh"
#include "lce_gemm.cuh"
#include "lce_rows.cuh"

using namespace lce;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSms = 256;              // bound used to size the (m, l) partials
// Vocab rows per backward chunk: big enough that the per-chunk launch
// overheads and dH-accumulator passes are small, small enough that a chunk's
// G and W rows stay largely L2-resident (6144 measured best of 2048..12288 on
// all four bf16 workloads).
constexpr int64_t kDefaultVocabChunk = 6144;
// G chunk buffers: three for a plain backward (chunk j is read while chunk
// j+1 is written, and the launch after may already write chunk j+2 while
// chunk j's last tiles run); four with a fused optimizer, whose dW tiles of
// chunk j run one launch later (see run_rows).
constexpr int kGBuffers = 3;
constexpr int kGBuffersOpt = 4;
constexpr int kMaxGBuffers = 4;

inline bool has_optim(const lce_args_t *a) { return a->optim && a->optim->kind != LCE_OPT_NONE; }

thread_local int t_last_cuda = 0;
std::atomic<int64_t> g_launches{0};
std::mutex g_mu;

struct DevInfo {
    bool ready = false;
    int sms = 0, major = 0, minor = 0;
};
DevInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// ----------------------------------------------------------------- profiling

struct PhaseRec {
    int phase;
    cudaEvent_t a, b;
    int64_t launches;
};
struct Profiler {
    bool on = false;
    std::vector<PhaseRec> recs;
    int64_t *cur = nullptr;
};
thread_local Profiler t_prof;

struct PhaseScope {
    cudaStream_t s;
    PhaseRec rec{};
    bool live = false;
    int64_t launches = 0;
    PhaseScope(int phase, cudaStream_t st) : s(st) {
        if (!t_prof.on) return;
        rec.phase = phase;
        if (cudaEventCreate(&rec.a) != cudaSuccess) return;
        if (cudaEventCreate(&rec.b) != cudaSuccess) {
            cudaEventDestroy(rec.a);
            return;
        }
        cudaEventRecord(rec.a, s);
        live = true;
        t_prof.cur = &launches;
    }
    ~PhaseScope() {
        if (!live) return;
        cudaEventRecord(rec.b, s);
        rec.launches = launches;
        t_prof.recs.push_back(rec);
        t_prof.cur = nullptr;
    }
};

inline void count_launch() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (t_prof.cur) ++*t_prof.cur;
}

// -------------------------------------------------------------------- device

lce_status_t device_info(DevInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &di = g_dev[dev];
    if (!di.ready) {
        cudaDeviceProp p;
        e = cudaGetDeviceProperties(&p, dev);
        if (e != cudaSuccess) {
            t_last_cuda = e;
            return LCE_ERR_CUDA;
        }
        di.sms = p.multiProcessorCount;
        di.major = p.major;
        di.minor = p.minor;
        if (!(di.major == 10 && di.minor == 3) || di.sms > kMaxSms) return LCE_ERR_DEVICE;
        const void *gemms[] = {(const void *)k_gemm<KIND_LSE>, (const void *)k_gemm<KIND_BWD>,
                               (const void *)k_gemm<KIND_BWD_OPT>};
        for (const void *f : gemms) {
            e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
            if (e != cudaSuccess) {
                t_last_cuda = e;
                return LCE_ERR_CUDA;
            }
        }
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
                t_last_cuda = e != cudaSuccess ? e : cudaErrorNotSupported;
                return LCE_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        di.ready = true;
    }
    *out = &di;
    return LCE_OK;
}

// 2-D bf16 tensor map over a row-major [outer][inner] array, 128-byte swizzle.
bool encode_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Map used by bulk tensor stores from the epilogue: box {32, 32} over a
// row-major [outer][inner] array of bf16 (64-byte swizzle) or fp32 (128-byte
// swizzle), matching the staging layout the epilogue writes.
bool encode_store_map(CUtensorMap *m, const void *base, bool fp32, uint64_t inner, uint64_t outer) {
    const uint64_t elt = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * elt};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D bf16 map over the same row-major [outer][inner] array for MN-major
// operand tiles: dims {64, outer, inner/64} with strides {row, 128 bytes}, so
// one box {64, box_rows, box_blocks} lands as box_blocks consecutive
// {box_rows x 128-byte} blocks, the layout the MN-major descriptors read.
// Only valid when inner is a multiple of 64 (a partial block would read into
// the next row instead of being zero-filled).
bool encode_map_mn3(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_rows,
                    uint32_t box_blocks) {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kAtom), outer, inner / kAtom};
    cuuint64_t strides[2] = {inner * 2, static_cast<cuuint64_t>(kAtom) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kAtom), box_rows, box_blocks};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Fused-optimizer boxes {16, 32} over a row-major [V][d] array: fp32 with
// 64-byte swizzle, or bf16 with 32-byte swizzle (the layouts the optimizer
// epilogue reads and writes).
bool encode_opt_map(CUtensorMap *m, const void *base, bool fp32, uint64_t d, uint64_t V) {
    const uint64_t elt = fp32 ? 4 : 2;
    cuuint64_t dims[2] = {d, V};
    cuuint64_t strides[1] = {d * elt};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          fp32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ----------------------------------------------------------------- workspace

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Row gather (lce_args_t.row_gather): the GEMMs read bf16 H's valid rows
// themselves (TMA gather4 through the compaction index) instead of a
// compacted copy Hc; only when d is a whole number of 256-column tiles, so
// that no gather4 ever starts outside H. Off by default: on this part it is
// several times slower than the copy kernel plus tiled loads (each gather4
// moves 512 bytes, 32 per stage per CTA), and saves only the N_pad*d*2-byte
// copy.
inline bool row_gather_ok(lce_dtype_t dt, int64_t d) { return dt == LCE_BF16 && d % kBN == 0; }

struct Layout {
    bool gather = false;
    int64_t N_pad = 0, Vc = 0, part_rows = 0;
    size_t idx = 0, inv = 0, counters = 0, tc = 0, z = 0, lse2 = 0, loss_rows = 0, part = 0, Hc = 0, Hc_lo = 0,
           W_hi = 0, W_lo = 0, G = 0, G_lo = 0, dHacc = 0, gcount = 0, lpart = 0, total = 0;
};

// Every operand the tensor cores read is bf16. fp32 inputs are carried as bf16
// hi/lo pairs (Hc/Hc_lo, W_hi/W_lo, G/G_lo), so the fp32 path also holds a
// split copy of W (4*V*d bytes).
Layout make_layout(int64_t N, int64_t d, int64_t V, lce_dtype_t dt, int64_t Vc, bool backward, int n_tc = 1,
                   int n_gbuf = kGBuffers, bool gather = false) {
    Layout L;
    const bool split = dt == LCE_FP32;
    L.N_pad = (N + kPairM - 1) / kPairM * kPairM;
    L.Vc = Vc;
    L.gather = gather && row_gather_ok(dt, d);
    L.part_rows = lse_partial_rows(static_cast<int>(L.N_pad), kMaxSms / 2);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += up256(bytes);
        return at;
    };
    L.idx = take(L.N_pad * 4);   // padded rows get an index too (row gather)
    L.inv = take(N * 4);
    L.counters = take(64);
    L.tc = take(L.N_pad * 4);
    L.z = take(L.N_pad * 4);
    L.lse2 = take(L.N_pad * 4);
    L.loss_rows = take(L.N_pad * 4);
    L.part = take(L.part_rows * 8);
    if (!L.gather) L.Hc = take(L.N_pad * d * 2);
    if (split) {
        L.Hc_lo = take(L.N_pad * d * 2);
        L.W_hi = take(static_cast<size_t>(V) * d * 2);
        L.W_lo = take(static_cast<size_t>(V) * d * 2);
    }
    if (backward) {
        L.G = take(n_gbuf * L.N_pad * Vc * 2);
        if (split) L.G_lo = take(n_gbuf * L.N_pad * Vc * 2);
        L.dHacc = take(L.N_pad * d * 4);
    }
    L.gcount = take(64);               // valid count of the whole call (token chunks)
    L.lpart = take(size_t(n_tc) * 8);  // per-token-chunk loss sums
    L.total = o;
    return L;
}

// Rows per token chunk: all N unless the caller capped it.
int64_t token_rows(int64_t N, int64_t token_chunk) { return token_chunk > 0 && token_chunk < N ? token_chunk : N; }

// Vocab rows per backward chunk: the caller's, else the default size spread
// evenly over the chunks it needs (rounded up to 256-row tiles), so that the
// last chunk is not a sliver (e.g. V = 32000: 6 chunks of 5376 instead of
// five of 6144 and one of 1280; 2% faster on that workload).
int64_t pick_chunk(int64_t V, int64_t requested) {
    const int64_t vpad = (V + kBN - 1) / kBN * kBN;
    int64_t c = requested;
    if (c <= 0) {
        const int64_t n = (V + kDefaultVocabChunk - 1) / kDefaultVocabChunk;
        c = ((V + n - 1) / n + kBN - 1) / kBN * kBN;
    }
    return c < vpad ? c : vpad;
}

lce_status_t check_args(const lce_args_t *a) {
    if (!a) return LCE_ERR_NULL;
    if (a->dtype != LCE_BF16 && a->dtype != LCE_FP32) return LCE_ERR_DTYPE;
    if (!a->H || !a->W || !a->targets) return LCE_ERR_NULL;
    // dH and dW together, or neither; with a fused optimizer dH alone
    if (has_optim(a) ? !a->dH : (a->dH == nullptr) != (a->dW == nullptr)) return LCE_ERR_NULL;
    if (a->lse_in ? !a->dH : !a->loss) return LCE_ERR_NULL;   // backward-only needs grads; forward needs loss
    if (a->N < 1 || a->N >= (int64_t(1) << 31) || a->d < 1 || a->d > 65536 || a->V < 1 ||
        a->V >= (int64_t(1) << 31))
        return LCE_ERR_SHAPE;
    if (a->vocab_chunk < 0 || (a->vocab_chunk > 0 && (a->vocab_chunk % kBN) != 0) ||
        a->vocab_chunk > (int64_t(1) << 20) || a->token_chunk < 0)
        return LCE_ERR_SHAPE;
    if (a->d % 8) return LCE_ERR_ALIGN;   // bf16 rows (operands or their split copies) of 16-byte multiples
    if (a->row_gather && !row_gather_ok(a->dtype, a->d)) return LCE_ERR_ARG;
    // a bf16 dW is written once per element: bf16 inputs, no accumulation, one token chunk
    if (a->dW_bf16 && (!a->dW || a->dtype != LCE_BF16 || a->accumulate_dW ||
                       (a->token_chunk > 0 && a->token_chunk < a->N)))
        return LCE_ERR_ARG;
    auto mis = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (mis(a->H) || mis(a->W) || (a->dH && mis(a->dH)) || (a->dW && mis(a->dW)) ||
        (a->workspace && mis(a->workspace)))
        return LCE_ERR_ALIGN;
    if (a->optim) {
        const lce_optim_t *o = a->optim;
        if (o->kind != LCE_OPT_NONE && o->kind != LCE_OPT_SGD && o->kind != LCE_OPT_ADAMW) return LCE_ERR_ARG;
        if (o->kind != LCE_OPT_NONE) {
            // the update consumes the gradient of the whole call: no dW output,
            // no accumulation into one, no token chunks
            if (!a->dH) return LCE_ERR_NULL;
            if (a->dW || a->accumulate_dW || token_rows(a->N, a->token_chunk) != a->N) return LCE_ERR_ARG;
            if (o->master_W && a->dtype != LCE_BF16) return LCE_ERR_ARG;
            if (!(o->lr >= 0.f) || !(o->weight_decay >= 0.f) || o->step < 1) return LCE_ERR_ARG;
            if (o->kind == LCE_OPT_ADAMW) {
                if (!o->exp_avg || !o->exp_avg_sq) return LCE_ERR_NULL;
                if (!(o->beta1 >= 0.f && o->beta1 < 1.f && o->beta2 >= 0.f && o->beta2 < 1.f && o->eps > 0.f))
                    return LCE_ERR_ARG;
            } else {
                if (!(o->momentum >= 0.f)) return LCE_ERR_ARG;
                if (o->momentum != 0.f && !o->exp_avg) return LCE_ERR_NULL;
            }
            if ((o->master_W && mis(o->master_W)) || (o->exp_avg && mis(o->exp_avg)) ||
                (o->exp_avg_sq && mis(o->exp_avg_sq)))
                return LCE_ERR_ALIGN;
        }
    }
    return LCE_OK;
}

struct WsGuard {
    void *p = nullptr;
    cudaStream_t s = nullptr;
    bool owned = false;
    ~WsGuard() {
        if (owned && p) cudaFreeAsync(p, s);
    }
};

#define LCE_CHECK_LAUNCH()                     \
    do {                                       \
        count_launch();                        \
        cudaError_t e_ = cudaGetLastError();   \
        if (e_ != cudaSuccess) {               \
            t_last_cuda = e_;                  \
            return LCE_ERR_CUDA;               \
        }                                      \
    } while (0)

// One token chunk of a call: rows [r0, r0 + a->N) of the caller's arrays
// (a is already offset to them), normalised by *nv_norm, its loss sum into
// *lpart, dW added into (acc_dw) or written.
struct RowsCtx {
    const int *nv_norm;   // nullptr: this chunk's own valid count
    double *lpart;
    bool acc_dw;
    bool split_w;         // split an fp32 W into bf16 hi/lo (first chunk only)
};

template <typename T>
lce_status_t run_rows(const lce_args_t *a, const DevInfo &di, uint8_t *base, const Layout &L, int64_t Vc,
                      const RowsCtx &ctx) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(a->stream);
    const bool backward = a->dH != nullptr;
    const bool split = a->dtype == LCE_FP32;
    const int N = static_cast<int>(a->N), d = static_cast<int>(a->d), V = static_cast<int>(a->V);
    auto bf = [&](size_t off) { return reinterpret_cast<__nv_bfloat16 *>(base + off); };
    int *idx = reinterpret_cast<int *>(base + L.idx);
    int *inv = reinterpret_cast<int *>(base + L.inv);
    int *counters = reinterpret_cast<int *>(base + L.counters);
    int *tc = reinterpret_cast<int *>(base + L.tc);
    float *z = reinterpret_cast<float *>(base + L.z);
    float *lse2 = reinterpret_cast<float *>(base + L.lse2);
    float *loss_rows = reinterpret_cast<float *>(base + L.loss_rows);
    float2 *part = reinterpret_cast<float2 *>(base + L.part);
    __nv_bfloat16 *Hc = L.gather ? nullptr : bf(L.Hc);
    __nv_bfloat16 *Hc_lo = split ? bf(L.Hc_lo) : nullptr;
    const __nv_bfloat16 *W_hi = split ? bf(L.W_hi) : static_cast<const __nv_bfloat16 *>(a->W);
    const __nv_bfloat16 *W_lo = split ? bf(L.W_lo) : W_hi;
    __nv_bfloat16 *G = backward ? bf(L.G) : nullptr;
    __nv_bfloat16 *G_lo = backward && split ? bf(L.G_lo) : G;
    float *dHacc = backward ? reinterpret_cast<float *>(base + L.dHacc) : nullptr;
    const __nv_bfloat16 *Hc_lo_or_hi = split ? Hc_lo : Hc;
    // row gather: one map over the caller's H with a one-row box
    CUtensorMap h_rows;
    memset(&h_rows, 0, sizeof(h_rows));
    if (L.gather && !encode_map(&h_rows, a->H, d, N, kBK, 1)) return LCE_ERR_CUDA;

    // K-major operand maps (box 64 x rows) and MN-major ones (box 64 x 64)
    GemmMaps maps_lse;
    memset(&maps_lse, 0, sizeof(maps_lse));
    {
        OperandMaps &o = maps_lse.t[map_slot(T_LSE)];
        if (L.gather) {
            o.A[0] = o.A[1] = h_rows;
        } else if (!encode_map(&o.A[0], Hc, d, L.N_pad, kBK, kBM) ||
                   !encode_map(&o.A[1], Hc_lo_or_hi, d, L.N_pad, kBK, kBM)) {
            return LCE_ERR_CUDA;
        }
        if (!encode_map(&o.B[0], W_hi, d, V, kBK, kHalfN) || !encode_map(&o.B[1], W_lo, d, V, kBK, kHalfN))
            return LCE_ERR_CUDA;
    }

    GemmArgs ga{};
    ga.counters = counters;
    ga.nv_norm = ctx.nv_norm ? ctx.nv_norm : counters;
    ga.d = d;
    ga.V = V;
    const int pairs = di.sms / 2;          // one CTA pair per two SMs
    const int grid = 2 * pairs;
    ga.num_pairs = pairs;
    ga.nseg = split ? 3 : 1;
    ga.tc = tc;
    ga.gather = L.gather ? 1 : 0;
    ga.idx = idx;
    ga.grad_scale = a->grad_scale == 0.f ? 1.f : a->grad_scale;
    ga.grad_ptr = a->grad_loss;
    const int n_tiles_v = cdiv(V, kBN);

    {
        PhaseScope ph(0, st);
        k_compact<<<1, kCompactThreads, 0, st>>>(a->targets, N, a->ignore_index, a->V, idx, inv, counters, a->lse);
        LCE_CHECK_LAUNCH();
        const int ggrid = static_cast<int>(L.N_pad < 4 * di.sms * 8 ? L.N_pad : 4 * di.sms * 8);
        k_gather<T><<<ggrid, 256, 0, st>>>(static_cast<const T *>(a->H), a->targets, d, a->V, idx, counters, Hc,
                                           Hc_lo, tc, z);
        LCE_CHECK_LAUNCH();
        if (split && ctx.split_w) {
            k_split_rows<<<4 * di.sms, 256, 0, st>>>(static_cast<const float *>(a->W), static_cast<size_t>(V) * d,
                                                     bf(L.W_hi), bf(L.W_lo));
            LCE_CHECK_LAUNCH();
        }
    }
    if (a->lse_in) {
        // backward from a stored lse: no forward pass
        PhaseScope ph(2, st);
        k_lse_from_input<<<static_cast<int>(L.N_pad / 256 + 1), 256, 0, st>>>(a->lse_in, idx, counters, lse2);
        LCE_CHECK_LAUNCH();
    } else {
        {
            PhaseScope ph(1, st);
            GemmArgs g = ga;
            g.z = z;
            g.part = part;
            k_gemm<KIND_LSE><<<grid, kThreads, kGemmSmem, st>>>(maps_lse, g);
            LCE_CHECK_LAUNCH();
        }
        PhaseScope ph(2, st);
        k_lse_merge<<<static_cast<int>(L.N_pad / 256 + 1), 256, 0, st>>>(part, counters, n_tiles_v, pairs, z, lse2,
                                                                         loss_rows, idx, a->lse);
        LCE_CHECK_LAUNCH();
        k_loss_partial<<<1, 1024, 0, st>>>(loss_rows, counters, ctx.lpart);
        LCE_CHECK_LAUNCH();
    }
    if (!backward) return LCE_OK;

    // Backward. Plain: launch j runs the G tiles of chunk j+1 (writing G
    // buffer (j+1)%3) and dW/dH of chunk j (reading buffer j%3); launch j = -1
    // only fills G of chunk 0 and the last launch has no next chunk. Launches
    // after the first are programmatic dependents of their predecessor: their
    // CTAs start as the predecessor's finish, and wait for it
    // (griddepcontrol.wait) before their dW/dH tiles. A launch signals its own
    // dependent only after that wait, so launch j+1 (writing buffer
    // (j+2)%3 = (j-1)%3) cannot start before launch j-1, the last reader of
    // that buffer, has completed.
    // With a fused optimizer the dW tiles of chunk j (which rewrite W rows of
    // chunk j) move to launch j+1, after its wait: launch j, whose dH tiles
    // are the last readers of those rows, has completed by then. Launch j
    // then reads buffers j%4 (dH) and (j-1)%4 (dW) while writing (j+1)%4, and
    // its dependent writes (j+2)%4 = (j-2)%4, last read in launch j-1.
    const bool opt = has_optim(a);
    const int nbuf = opt ? kGBuffersOpt : kGBuffers;
    const size_t gbuf = static_cast<size_t>(L.N_pad) * Vc;   // elements per G buffer
    const bool mn3d_d = (d % kAtom) == 0;
    OperandMaps dh_maps[kMaxGBuffers], dw_maps[kMaxGBuffers];
    memset(dh_maps, 0, sizeof(dh_maps));
    memset(dw_maps, 0, sizeof(dw_maps));
    for (int b = 0; b < nbuf; ++b) {
        const __nv_bfloat16 *Gb = G + b * gbuf;
        const __nv_bfloat16 *Gb_lo = G_lo + b * gbuf;
        OperandMaps &dh = dh_maps[b];
        OperandMaps &dw = dw_maps[b];
        if (!encode_map(&dh.A[0], Gb, Vc, L.N_pad, kBK, kBM) || !encode_map(&dh.A[1], Gb_lo, Vc, L.N_pad, kBK, kBM) ||
            !encode_map_mn3(&dw.A[0], Gb, Vc, L.N_pad, kBK, kBM / kAtom) ||
            !encode_map_mn3(&dw.A[1], Gb_lo, Vc, L.N_pad, kBK, kBM / kAtom))
            return LCE_ERR_CUDA;
        if (L.gather) {
            if (!encode_map_mn3(&dh.B[0], W_hi, d, V, kBK, kHalfN / kAtom) ||
                !encode_map_mn3(&dh.B[1], W_lo, d, V, kBK, kHalfN / kAtom))
                return LCE_ERR_CUDA;
            dw.B[0] = dw.B[1] = h_rows;
        } else if (mn3d_d) {
            if (!encode_map_mn3(&dh.B[0], W_hi, d, V, kBK, kHalfN / kAtom) ||
                !encode_map_mn3(&dh.B[1], W_lo, d, V, kBK, kHalfN / kAtom) ||
                !encode_map_mn3(&dw.B[0], Hc, d, L.N_pad, kBK, kHalfN / kAtom) ||
                !encode_map_mn3(&dw.B[1], Hc_lo_or_hi, d, L.N_pad, kBK, kHalfN / kAtom))
                return LCE_ERR_CUDA;
        } else if (!encode_map(&dh.B[0], W_hi, d, V, kAtom, kBK) || !encode_map(&dh.B[1], W_lo, d, V, kAtom, kBK) ||
                   !encode_map(&dw.B[0], Hc, d, L.N_pad, kAtom, kBK) ||
                   !encode_map(&dw.B[1], Hc_lo_or_hi, d, L.N_pad, kAtom, kBK)) {
            return LCE_ERR_CUDA;
        }
    }
    CUtensorMap st_g[kMaxGBuffers][2], st_dw, st_dh;
    memset(&st_dw, 0, sizeof(st_dw));
    for (int b = 0; b < nbuf; ++b)
        if (!encode_store_map(&st_g[b][0], G + b * gbuf, false, Vc, L.N_pad) ||
            !encode_store_map(&st_g[b][1], G_lo + b * gbuf, false, Vc, L.N_pad))
            return LCE_ERR_CUDA;
    if ((a->dW && !encode_store_map(&st_dw, a->dW, !a->dW_bf16, d, V)) ||
        !encode_store_map(&st_dh, dHacc, true, d, L.N_pad))
        return LCE_ERR_CUDA;

    OptArgs oa{};
    CUtensorMap opt_maps[4];   // m, v, fp32 weights, bf16 W
    memset(opt_maps, 0, sizeof(opt_maps));
    if (opt) {
        const lce_optim_t *o = a->optim;
        const bool use_m = o->kind == LCE_OPT_ADAMW || o->momentum != 0.f;
        const float *w32 = o->master_W ? o->master_W : (a->dtype == LCE_FP32 ? static_cast<const float *>(a->W) : nullptr);
        const bool s32 = !o->state_bf16;
        if ((use_m && !encode_opt_map(&opt_maps[0], o->exp_avg, s32, d, V)) ||
            (o->kind == LCE_OPT_ADAMW && !encode_opt_map(&opt_maps[1], o->exp_avg_sq, s32, d, V)) ||
            (w32 && !encode_opt_map(&opt_maps[2], w32, true, d, V)) ||
            (a->dtype == LCE_BF16 && !encode_opt_map(&opt_maps[3], a->W, false, d, V)))
            return LCE_ERR_CUDA;
        oa.kind = o->kind == LCE_OPT_ADAMW ? OPT_ADAMW : OPT_SGD;
        oa.first = o->step == 1;
        oa.lr = o->lr;
        oa.wd = o->weight_decay;
        oa.momentum = o->momentum;
        oa.beta1 = o->beta1;
        oa.beta2 = o->beta2;
        oa.eps = o->eps;
        if (oa.kind == OPT_ADAMW) {
            const double t = static_cast<double>(o->step);
            oa.step_size = static_cast<float>(o->lr / (1.0 - pow(static_cast<double>(o->beta1), t)));
            oa.inv_bc2_sqrt = static_cast<float>(1.0 / sqrt(1.0 - pow(static_cast<double>(o->beta2), t)));
        }
        oa.W = const_cast<void *>(a->W);
        oa.w_fp32 = a->dtype == LCE_FP32;
        oa.master = o->master_W;
        oa.m = o->exp_avg;
        oa.v = o->exp_avg_sq;
        oa.s16 = o->state_bf16 ? 1 : 0;
    }

    const int n_chunks = static_cast<int>((a->V + Vc - 1) / Vc);
    auto chunk_len = [&](int c) { return static_cast<int>(a->V - c * Vc < Vc ? a->V - c * Vc : Vc); };
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    void (*bwd_kernel)(const GemmMaps, const GemmArgs) = opt ? k_gemm<KIND_BWD_OPT> : k_gemm<KIND_BWD>;
    {
        PhaseScope ph(3, st);
        const int last = opt ? n_chunks : n_chunks - 1;
        for (int j = -1; j <= last; ++j) {
            const int cw = opt ? j - 1 : j;   // chunk whose dW tiles this launch runs
            GemmArgs g = ga;
            g.lse2 = lse2;
            g.has_cur = j >= 0 && j < n_chunks;
            g.has_next = j + 1 < n_chunks;
            g.has_dw = cw >= 0 && cw < n_chunks;
            if (g.has_cur) {
                g.v0 = static_cast<int>(j * Vc);
                g.vlen = chunk_len(j);
            }
            if (g.has_next) {
                g.v0n = static_cast<int>((j + 1) * Vc);
                g.vlenn = chunk_len(j + 1);
            }
            if (g.has_dw) {
                g.v0w = static_cast<int>(cw * Vc);
                g.vlenw = chunk_len(cw);
            }
            g.mn3d = 1 | (mn3d_d ? 6 : 0);
            g.dW = static_cast<float *>(a->dW);   // bf16 rows when dw_bf16
            g.dw_bf16 = a->dW_bf16 ? 1 : 0;
            g.acc_dw = ctx.acc_dw ? 1 : 0;
            g.dH_acc = dHacc;
            g.acc_dh = j > 0 ? 1 : 0;
            g.opt = oa;
            // every slot holds a valid map (buffer 0 where a tile type is absent)
            GemmMaps mp;
            mp.t[map_slot(T_G)] = maps_lse.t[map_slot(T_LSE)];
            mp.t[map_slot(T_DH)] = dh_maps[g.has_cur ? j % nbuf : 0];
            mp.t[map_slot(T_DW)] = dw_maps[g.has_dw ? cw % nbuf : 0];
            mp.st_g[0] = st_g[g.has_next ? (j + 1) % nbuf : 0][0];
            mp.st_g[1] = st_g[g.has_next ? (j + 1) % nbuf : 0][1];
            mp.st_dw = st_dw;
            mp.st_dh = st_dh;
            mp.opt_m = opt_maps[0];
            mp.opt_v = opt_maps[1];
            mp.opt_w32 = opt_maps[2];
            mp.opt_w16 = opt_maps[3];
            if (j < 0) {
                bwd_kernel<<<grid, kThreads, kGemmSmem, st>>>(mp, g);
            } else {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(grid);
                cfg.blockDim = dim3(kThreads);
                cfg.dynamicSmemBytes = kGemmSmem;
                cfg.stream = st;
                cfg.attrs = pdl;
                cfg.numAttrs = 1;
                cudaError_t e = cudaLaunchKernelEx(&cfg, bwd_kernel, mp, g);
                if (e != cudaSuccess) {
                    t_last_cuda = e;
                    return LCE_ERR_CUDA;
                }
            }
            LCE_CHECK_LAUNCH();
        }
    }
    {
        PhaseScope ph(4, st);
        const int sgrid = N < 8 * di.sms ? N : 8 * di.sms;
        k_dh_scatter<T><<<sgrid, 256, 0, st>>>(dHacc, inv, N, d, static_cast<T *>(a->dH));
        LCE_CHECK_LAUNCH();
    }
    return LCE_OK;
}

template <typename T>
lce_status_t run_typed(const lce_args_t *a, const DevInfo &di) {
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(a->stream);
    const bool backward = a->dH != nullptr;
    const int64_t Vc = pick_chunk(a->V, a->vocab_chunk);
    const int64_t C = token_rows(a->N, a->token_chunk);
    const int n_tc = static_cast<int>((a->N + C - 1) / C);
    const Layout L = make_layout(C, a->d, a->V, a->dtype, Vc, backward, n_tc,
                                 has_optim(a) ? kGBuffersOpt : kGBuffers, a->row_gather != 0);

    WsGuard ws;
    ws.s = st;
    if (a->workspace) {
        if (a->workspace_bytes < L.total) return LCE_ERR_WORKSPACE;
        ws.p = a->workspace;
    } else {
        cudaError_t e = cudaMallocAsync(&ws.p, L.total, st);
        if (e != cudaSuccess) {
            t_last_cuda = e;
            return LCE_ERR_CUDA;
        }
        ws.owned = true;
    }
    uint8_t *base = static_cast<uint8_t *>(ws.p);
    int *gcount = reinterpret_cast<int *>(base + L.gcount);
    double *lpart = reinterpret_cast<double *>(base + L.lpart);
    const bool chunked = n_tc > 1;
    if (chunked) {
        // the normaliser is the valid count of all N rows, known before any chunk
        PhaseScope ph(0, st);
        k_count_valid<<<1, 1024, 0, st>>>(a->targets, static_cast<int>(a->N), a->ignore_index, gcount);
        LCE_CHECK_LAUNCH();
    }
    const size_t elt = a->dtype == LCE_BF16 ? 2 : 4;
    for (int c = 0; c < n_tc; ++c) {
        const int64_t r0 = c * C;
        lce_args_t ac = *a;
        ac.N = (a->N - r0 < C) ? a->N - r0 : C;
        ac.H = static_cast<const uint8_t *>(a->H) + r0 * a->d * elt;
        ac.targets = a->targets + r0;
        if (a->dH) ac.dH = static_cast<uint8_t *>(a->dH) + r0 * a->d * elt;
        if (a->lse) ac.lse = a->lse + r0;
        if (a->lse_in) ac.lse_in = a->lse_in + r0;
        RowsCtx ctx;
        ctx.nv_norm = chunked ? gcount : nullptr;
        ctx.lpart = lpart + c;
        ctx.acc_dw = a->accumulate_dW || c > 0;
        ctx.split_w = c == 0;
        const lce_status_t s = run_rows<T>(&ac, di, base, L, Vc, ctx);
        if (s != LCE_OK) return s;
    }
    if (!a->lse_in) {
        PhaseScope ph(2, st);
        const int *nvn = chunked ? gcount : reinterpret_cast<const int *>(base + L.counters);
        k_loss_final<<<1, 32, 0, st>>>(lpart, n_tc, nvn, a->loss);
        LCE_CHECK_LAUNCH();
    }
    return LCE_OK;
}

// ------------------------------------------------------ allocation-free entry
//
// Scratch for lce_forward_noalloc: a fixed device array that every GPU loading
// this library holds until the process exits. Its host-side name is only a
// stand-in; the device address is looked up once per device.
constexpr int64_t kNoAllocMaxN = 4096;
constexpr int64_t kNoAllocMaxD = 2048;
constexpr size_t kNoAllocScratchBytes = size_t(21) << 20;   // 21 MiB: bf16 Hc of 4096 x 2048 + row buffers

void *g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch on the current device, looked up the
// first time each device is seen (with that device current).
lce_status_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            t_last_cuda = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return LCE_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return LCE_OK;
}

}  // namespace

extern "C" {

lce_status_t lce_run(const lce_args_t *a) {
    lce_status_t s = check_args(a);
    if (s != LCE_OK) return s;
    DevInfo *di = nullptr;
    s = device_info(&di);
    if (s != LCE_OK) return s;
    return a->dtype == LCE_BF16 ? run_typed<__nv_bfloat16>(a, *di) : run_typed<float>(a, *di);
}

lce_status_t lce_forward(const void *H, const void *W, const int64_t *targets, int64_t ignore_index, int64_t N,
                         int64_t d, int64_t V, float *loss, lce_stream_t stream) {
    lce_args_t a{};
    a.dtype = LCE_BF16;
    a.H = H;
    a.W = W;
    a.targets = targets;
    a.ignore_index = ignore_index;
    a.N = N;
    a.d = d;
    a.V = V;
    a.loss = loss;
    a.stream = stream;
    return lce_run(&a);
}

lce_status_t lce_forward_backward(const void *H, const void *W, const int64_t *targets, int64_t ignore_index,
                                  int64_t N, int64_t d, int64_t V, float *loss, void *dH, float *dW,
                                  lce_stream_t stream) {
    if (!dH || !dW) return LCE_ERR_NULL;
    lce_args_t a{};
    a.dtype = LCE_BF16;
    a.H = H;
    a.W = W;
    a.targets = targets;
    a.ignore_index = ignore_index;
    a.N = N;
    a.d = d;
    a.V = V;
    a.loss = loss;
    a.dH = dH;
    a.dW = dW;
    a.stream = stream;
    return lce_run(&a);
}

lce_status_t lce_backward(const void *H, const void *W, const int64_t *targets, int64_t ignore_index, int64_t N,
                          int64_t d, int64_t V, const float *lse, const float *grad_loss, void *dH, float *dW,
                          lce_stream_t stream) {
    if (!lse || !dH || !dW) return LCE_ERR_NULL;
    lce_args_t a{};
    a.dtype = LCE_BF16;
    a.H = H;
    a.W = W;
    a.targets = targets;
    a.ignore_index = ignore_index;
    a.N = N;
    a.d = d;
    a.V = V;
    a.dH = dH;
    a.dW = dW;
    a.lse_in = lse;
    a.grad_loss = grad_loss;
    a.stream = stream;
    return lce_run(&a);
}

lce_status_t lce_compact(const int64_t *targets, int64_t N, int64_t ignore_index, int64_t V, int32_t *idx,
                         int32_t *inv, int32_t *counts, lce_stream_t stream) {
    if (!targets || !idx || !inv || !counts) return LCE_ERR_NULL;
    if (N < 1 || N >= (int64_t(1) << 31) || V < 1 || V >= (int64_t(1) << 31)) return LCE_ERR_SHAPE;
    DevInfo *di = nullptr;
    lce_status_t s = device_info(&di);
    if (s != LCE_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    PhaseScope ph(0, st);
    k_compact<<<1, kCompactThreads, 0, st>>>(targets, static_cast<int>(N), ignore_index, V, idx, inv, counts,
                                             nullptr);
    LCE_CHECK_LAUNCH();
    return LCE_OK;
}

// ------------------------------------------------- input-embedding lookup

namespace {
struct EmbLayout {
    size_t kA, vA, kB, vB, hist, counts, partial, total;
};
EmbLayout emb_layout(int64_t N, int64_t d) {
    EmbLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o += up256(bytes);
        return at;
    };
    L.kA = take(N * 4);
    L.vA = take(N * 4);
    L.kB = take(N * 4);
    L.vB = take(N * 4);
    L.hist = take(static_cast<size_t>(kEmbBuckets) * kEmbMaxSortBlocks * 4);
    L.counts = take(16);
    L.partial = take(static_cast<size_t>(2 * emb_chunks_max(N)) * d * 4);
    L.total = o;
    return L;
}

lce_status_t check_emb(lce_dtype_t dtype, const void *a, const void *b, const int64_t *tokens, int64_t N, int64_t d,
                       int64_t V) {
    if (dtype != LCE_BF16 && dtype != LCE_FP32) return LCE_ERR_DTYPE;
    if (!a || !b || !tokens) return LCE_ERR_NULL;
    if (N < 1 || N >= (int64_t(1) << 31) || d < 1 || d > 65536 || V < 1 || V >= (int64_t(1) << 31))
        return LCE_ERR_SHAPE;
    if (d % 8 || (reinterpret_cast<uintptr_t>(a) & 15u) || (reinterpret_cast<uintptr_t>(b) & 15u))
        return LCE_ERR_ALIGN;
    return LCE_OK;
}
}  // namespace

lce_status_t lce_embedding_forward(lce_dtype_t dtype, const void *W, const int64_t *tokens, int64_t pad_id, int64_t N,
                                   int64_t d, int64_t V, void *E, lce_stream_t stream) {
    lce_status_t s = check_emb(dtype, W, E, tokens, N, d, V);
    if (s != LCE_OK) return s;
    DevInfo *di = nullptr;
    s = device_info(&di);
    if (s != LCE_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int rows_per_block = 256 / 32;
    const int64_t want = (N + rows_per_block - 1) / rows_per_block;
    const int grid = static_cast<int>(want < 8 * di->sms ? want : 8 * di->sms);
    if (dtype == LCE_BF16)
        k_emb_forward<__nv_bfloat16><<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(W), tokens, pad_id,
                                                            static_cast<int>(N), static_cast<int>(d), V,
                                                            static_cast<__nv_bfloat16 *>(E));
    else
        k_emb_forward<float><<<grid, 256, 0, st>>>(static_cast<const float *>(W), tokens, pad_id, static_cast<int>(N),
                                                   static_cast<int>(d), V, static_cast<float *>(E));
    LCE_CHECK_LAUNCH();
    return LCE_OK;
}

size_t lce_embedding_workspace_size(int64_t N, int64_t d) {
    if (N < 1 || N >= (int64_t(1) << 31) || d < 1 || d > 65536) return 0;
    return emb_layout(N, d).total;
}

namespace {
// dW fp32 (accumulate allowed) or bf16 (dw_bf16: each row's fp32 sum rounded
// once, overwritten)
lce_status_t emb_backward(lce_dtype_t dtype, const void *dE, const int64_t *tokens, int64_t pad_id, int64_t N,
                          int64_t d, int64_t V, void *dW, bool dw_bf16, int accumulate, void *workspace,
                          size_t workspace_bytes, lce_stream_t stream) {
    lce_status_t s = check_emb(dtype, dE, dW, tokens, N, d, V);
    if (s != LCE_OK) return s;
    const EmbLayout L = emb_layout(N, d);
    if (workspace && (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 15u)))
        return workspace_bytes < L.total ? LCE_ERR_WORKSPACE : LCE_ERR_ALIGN;
    DevInfo *di = nullptr;
    s = device_info(&di);
    if (s != LCE_OK) return s;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    WsGuard ws;
    ws.s = st;
    if (workspace) {
        ws.p = workspace;
    } else {
        cudaError_t e = cudaMallocAsync(&ws.p, L.total, st);
        if (e != cudaSuccess) {
            t_last_cuda = e;
            return LCE_ERR_CUDA;
        }
        ws.owned = true;
    }
    uint8_t *base = static_cast<uint8_t *>(ws.p);
    auto ip = [&](size_t off) { return reinterpret_cast<int *>(base + off); };
    int *counts = ip(L.counts);
    int *hist = ip(L.hist);
    float *partial = reinterpret_cast<float *>(base + L.partial);
    if (!accumulate) {
        // V*d fp32 elements, or the same bytes as half as many floats for bf16
        // (d % 8 == 0: a multiple of four floats either way)
        const size_t n = static_cast<size_t>(V) * d / (dw_bf16 ? 2 : 1);
        k_zero_f32<<<4 * di->sms, 256, 0, st>>>(static_cast<float *>(dW), n);
        LCE_CHECK_LAUNCH();
    }
    // group the valid positions by token: stable LSD radix passes, ping-pong
    // between the A and B key/position arrays (pass 0 reads the token ids)
    const int sblocks = emb_sort_blocks(N);
    const int span = static_cast<int>(emb_sort_span(N));
    const int passes = emb_radix_passes(V);
    int *keys[2] = {ip(L.kA), ip(L.kB)};
    int *vals[2] = {ip(L.vA), ip(L.vB)};
    for (int p = 0; p < passes; ++p) {
        EmbSortIn in{};
        in.t = tokens;
        in.keys = p ? keys[(p - 1) & 1] : nullptr;
        in.vals = p ? vals[(p - 1) & 1] : nullptr;
        in.pad_id = pad_id;
        in.V = V;
        in.first = p == 0;
        in.n = static_cast<int>(N);
        const int shift = p * kEmbRadixBits;
        k_emb_hist<<<sblocks, kEmbSortThreads, 0, st>>>(in, counts, span, shift, hist);
        LCE_CHECK_LAUNCH();
        k_emb_scatter<<<sblocks, kEmbSortThreads, 0, st>>>(in, counts, span, shift, hist, keys[p & 1], vals[p & 1]);
        LCE_CHECK_LAUNCH();
    }
    const int *skeys = keys[(passes - 1) & 1];
    const int *order = vals[(passes - 1) & 1];
    const unsigned slices = static_cast<unsigned>((d + kEmbSegCols - 1) / kEmbSegCols);
    const unsigned sum_slices = static_cast<unsigned>((d + kEmbSegSumCols - 1) / kEmbSegSumCols);
    const int64_t cmax = emb_chunks_max(N);
    const dim3 pgrid(static_cast<unsigned>(cmax < 8 * di->sms ? cmax : 8 * di->sms), sum_slices);
    const int acc = accumulate ? 1 : 0;
    const int di32 = static_cast<int>(d);
    auto segsum = [&](auto *out) {
        using O = std::remove_pointer_t<decltype(out)>;
        if (dtype == LCE_BF16)
            k_emb_segsum<__nv_bfloat16, O><<<pgrid, kEmbSegSumCols / 8, 0, st>>>(
                static_cast<const __nv_bfloat16 *>(dE), counts, skeys, order, di32, out, partial, acc);
        else
            k_emb_segsum<float, O><<<pgrid, kEmbSegSumCols / 8, 0, st>>>(static_cast<const float *>(dE), counts, skeys,
                                                                      order, di32, out, partial, acc);
    };
    const dim3 cgrid(static_cast<unsigned>(cmax < 4 * di->sms ? cmax : 4 * di->sms), slices);
    if (dw_bf16) {
        segsum(static_cast<__nv_bfloat16 *>(dW));
        LCE_CHECK_LAUNCH();
        k_emb_combine<__nv_bfloat16><<<cgrid, kEmbSegCols / 4, 0, st>>>(counts, skeys, di32,
                                                                        static_cast<__nv_bfloat16 *>(dW), partial, 0);
    } else {
        segsum(static_cast<float *>(dW));
        LCE_CHECK_LAUNCH();
        k_emb_combine<float><<<cgrid, kEmbSegCols / 4, 0, st>>>(counts, skeys, di32, static_cast<float *>(dW), partial,
                                                                acc);
    }
    LCE_CHECK_LAUNCH();
    return LCE_OK;
}
}  // namespace

lce_status_t lce_embedding_backward(lce_dtype_t dtype, const void *dE, const int64_t *tokens, int64_t pad_id,
                                    int64_t N, int64_t d, int64_t V, float *dW, int accumulate, void *workspace,
                                    size_t workspace_bytes, lce_stream_t stream) {
    return emb_backward(dtype, dE, tokens, pad_id, N, d, V, dW, false, accumulate, workspace, workspace_bytes, stream);
}

lce_status_t lce_embedding_backward_bf16(lce_dtype_t dtype, const void *dE, const int64_t *tokens, int64_t pad_id,
                                         int64_t N, int64_t d, int64_t V, void *dW, void *workspace,
                                         size_t workspace_bytes, lce_stream_t stream) {
    return emb_backward(dtype, dE, tokens, pad_id, N, d, V, dW, true, 0, workspace, workspace_bytes, stream);
}

size_t lce_workspace_size(int64_t N, int64_t d, int64_t V, lce_dtype_t dtype, int64_t vocab_chunk) {
    if (N < 1 || N >= (int64_t(1) << 31) || d < 1 || d > 65536 || V < 1 || V >= (int64_t(1) << 31)) return 0;
    if (dtype != LCE_BF16 && dtype != LCE_FP32) return 0;
    if (vocab_chunk < 0 || (vocab_chunk > 0 && vocab_chunk % kBN)) return 0;
    return make_layout(N, d, V, dtype, pick_chunk(V, vocab_chunk), true).total;
}

size_t lce_workspace_size_args(const lce_args_t *a) {
    if (!a || a->N < 1 || a->N >= (int64_t(1) << 31) || a->d < 1 || a->d > 65536 || a->V < 1 ||
        a->V >= (int64_t(1) << 31))
        return 0;
    if (a->dtype != LCE_BF16 && a->dtype != LCE_FP32) return 0;
    if (a->vocab_chunk < 0 || (a->vocab_chunk > 0 && a->vocab_chunk % kBN) || a->token_chunk < 0) return 0;
    const int64_t C = token_rows(a->N, a->token_chunk);
    const int n_tc = static_cast<int>((a->N + C - 1) / C);
    return make_layout(C, a->d, a->V, a->dtype, pick_chunk(a->V, a->vocab_chunk), a->dH != nullptr, n_tc,
                       has_optim(a) ? kGBuffersOpt : kGBuffers, a->row_gather != 0)
        .total;
}

lce_status_t lce_get_device_status(lce_stream_t stream, int32_t *bits) {
    if (!bits) return LCE_ERR_NULL;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    *bits = v;
    if (v & LCE_DEV_TARGET_RANGE) return LCE_ERR_TARGET_RANGE;
    if (v & LCE_DEV_TIMEOUT) return LCE_ERR_TIMEOUT;
    return LCE_OK;
}

const char *lce_status_string(lce_status_t s) {
    switch (s) {
        case LCE_OK: return "ok";
        case LCE_ERR_NULL: return "a required pointer is NULL";
        case LCE_ERR_SHAPE: return "N, d, V or vocab_chunk out of range";
        case LCE_ERR_ALIGN: return "pointer or row stride not 16-byte aligned";
        case LCE_ERR_DTYPE: return "unknown dtype";
        case LCE_ERR_CUDA: return "a CUDA call failed";
        case LCE_ERR_WORKSPACE: return "workspace smaller than lce_workspace_size()";
        case LCE_ERR_TARGET_RANGE: return "a non-ignored target is outside [0, V)";
        case LCE_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
        case LCE_ERR_DEVICE: return "the current device is not sm_103";
        case LCE_ERR_ARG: return "unsupported combination of options";
    }
    return "unknown status";
}

int lce_last_cuda_error(void) { return t_last_cuda; }

int64_t lce_launch_count(void) { return g_launches.load(); }

lce_status_t lce_profile_begin(void) {
    for (auto &r : t_prof.recs) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    t_prof.recs.clear();
    t_prof.on = true;
    return LCE_OK;
}

lce_status_t lce_profile_end(double *ms, int64_t *launches, int n) {
    t_prof.on = false;
    lce_status_t st = LCE_OK;
    for (int i = 0; i < n; ++i) {
        if (ms) ms[i] = 0.0;
        if (launches) launches[i] = 0;
    }
    for (auto &r : t_prof.recs) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
        if (e != cudaSuccess) {
            t_last_cuda = e;
            st = LCE_ERR_CUDA;
        } else if (r.phase < n) {
            if (ms) ms[r.phase] += t;
            if (launches) launches[r.phase] += r.launches;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    t_prof.recs.clear();
    return st;
}

lce_status_t lce_forward_noalloc(const void *H, const void *W, const int64_t *targets, int64_t ignore_index,
                                 int64_t N, int64_t d, int64_t V, float *loss, lce_stream_t stream) {
    if (!H || !W || !targets || !loss) return LCE_ERR_NULL;
    if (N < 1 || N > kNoAllocMaxN || d < 1 || d > kNoAllocMaxD || V < 1 || V >= (int64_t(1) << 31))
        return LCE_ERR_SHAPE;
    const Layout L = make_layout(N, d, V, LCE_BF16, pick_chunk(V, 0), false);
    if (L.total > kNoAllocScratchBytes) return LCE_ERR_SHAPE;
    DevInfo *di = nullptr;
    lce_status_t s = device_info(&di);
    if (s != LCE_OK) return s;
    void *scratch = nullptr;
    s = noalloc_scratch(&scratch);
    if (s != LCE_OK) return s;
    // The array keeps the previous call's contents; the compaction kernel
    // rewrites the counters, but they are cleared first so nothing can read a
    // stale valid-token count.
    cudaError_t e = cudaMemsetAsync(static_cast<uint8_t *>(scratch) + L.counters, 0, 64,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        t_last_cuda = e;
        return LCE_ERR_CUDA;
    }
    lce_args_t a{};
    a.dtype = LCE_BF16;
    a.H = H;
    a.W = W;
    a.targets = targets;
    a.ignore_index = ignore_index;
    a.N = N;
    a.d = d;
    a.V = V;
    a.loss = loss;
    a.workspace = scratch;
    a.workspace_bytes = kNoAllocScratchBytes;
    a.stream = stream;
    return lce_run(&a);
}

lce_status_t lce_selftest_wait_timeout(int64_t cycles, int32_t *gave_up, lce_stream_t stream) {
    if (!gave_up) return LCE_ERR_NULL;
    if (cycles < 1 || cycles > (int64_t(1) << 34)) return LCE_ERR_SHAPE;
    DevInfo *di = nullptr;
    lce_status_t s = device_info(&di);
    if (s != LCE_OK) return s;
    k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(cycles, gave_up);
    LCE_CHECK_LAUNCH();
    return LCE_OK;
}

int lce_version(void) { return 600; }

}  // extern "C"
