// Row-level (SIMT) kernels around the tensor-core passes: valid-token
// compaction, gather of the valid rows, log-sum-exp merge, the deterministic
// loss reduction and the final scatter of dH. All are HBM- or latency-bound.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "lce_gemm.cuh"

namespace lce {

constexpr int kCompactThreads = 1024;

// Dense ascending index list of the rows whose target is not ignore_index:
// one CTA sweeps the targets 1024 at a time; each warp takes a ballot of its
// valid lanes, __popc of the lower lanes gives the in-warp rank, and a scan
// over the 32 warp counts gives the warp offsets. The padding-aware valid mask
// of "为什么26万词表会卡死16GB显卡" (section 2.3 稀疏索引引擎), kept as an index
// list so the tensor-core passes see only dense rows.
//   idx[0..Nv)  ascending positions       inv[i]  compacted row or -1
//   counters[0] = Nv, counters[1] = number of non-ignored targets outside [0,V)
//   lse_user (optional) gets NaN on ignored rows.
__global__ void __launch_bounds__(kCompactThreads)
    k_compact(const int64_t *__restrict__ t, int N, int64_t ignore_index, int64_t V, int *__restrict__ idx,
              int *__restrict__ inv, int *__restrict__ counters, float *__restrict__ lse_user) {
    __shared__ int warp_incl[32];
    __shared__ int bad_total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) bad_total = 0;
    int running = 0, bad = 0;
    for (int base = 0; base < N; base += kCompactThreads) {
        const int i = base + threadIdx.x;
        const bool in = i < N;
        const int64_t ti = in ? t[i] : ignore_index;
        const bool valid = in && ti != ignore_index;
        bad += (valid && (ti < 0 || ti >= V)) ? 1 : 0;
        const unsigned m = __ballot_sync(0xffffffffu, valid);
        const int pre = __popc(m & ((1u << lane) - 1u));
        if (lane == 0) warp_incl[warp] = __popc(m);
        __syncthreads();
        if (warp == 0) {
            int v = warp_incl[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += n;
            }
            warp_incl[lane] = v;
        }
        __syncthreads();
        const int pos = running + (warp ? warp_incl[warp - 1] : 0) + pre;
        if (valid) idx[pos] = i;
        if (in) {
            inv[i] = valid ? pos : -1;
            if (lse_user && !valid) lse_user[i] = __int_as_float(0x7fc00000);
        }
        running += warp_incl[31];
        __syncthreads();
    }
    if (bad) atomicAdd(&bad_total, bad);
    __syncthreads();
    if (threadIdx.x == 0) {
        counters[0] = running;
        counters[1] = bad_total;
        if (bad_total) atomicOr(&g_status, DEV_TARGET_RANGE);
    }
}

// Hc[r] = H[idx[r]] for r < Nv, zero rows on [Nv, round_up(Nv, 256)) so the
// tensor-core passes can read whole 256-row pair blocks; tc[r] = target (or -1),
// z[r] = NaN until the logits pass finds the target column. bf16 rows are
// copied; fp32 rows are split into bf16 hi and lo parts (Hc, Hc_lo). With
// Hc == nullptr the GEMMs gather H's rows themselves: no rows are copied and
// idx[r] for the padded rows r in [Nv, round_up(Nv, 256)) is set to idx[0], a
// valid row (finite values; the padded rows' softmax gradient is zero).
__device__ __forceinline__ void gather8(const __nv_bfloat16 *src, __nv_bfloat16 *hi, __nv_bfloat16 *, bool live) {
    *reinterpret_cast<uint4 *>(hi) = live ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0, 0, 0, 0);
}
__device__ __forceinline__ void gather8(const float *src, __nv_bfloat16 *hi, __nv_bfloat16 *lo, bool live) {
    float h[8], l[8];
    if (live) {
        const float4 a = reinterpret_cast<const float4 *>(src)[0];
        const float4 b = reinterpret_cast<const float4 *>(src)[1];
        const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) split_bf16(x[j], h[j], l[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = l[j] = 0.f;
    }
    *reinterpret_cast<uint4 *>(hi) =
        make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
    *reinterpret_cast<uint4 *>(lo) =
        make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
}

template <typename T>
__global__ void __launch_bounds__(256)
    k_gather(const T *__restrict__ H, const int64_t *__restrict__ t, int d, int64_t V, int *__restrict__ idx,
             const int *__restrict__ counters, __nv_bfloat16 *__restrict__ Hc, __nv_bfloat16 *__restrict__ Hc_lo,
             int *__restrict__ tc, float *__restrict__ z) {
    const int nv = counters[0];
    const int rows = cdiv(nv, kPairM) * kPairM;
    const int groups = d / 8;   // d is a multiple of 8
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const bool live = r < nv;
        const int src_row = live ? idx[r] : 0;
        if (Hc) {
            const T *src = H + static_cast<size_t>(src_row) * d;
            __nv_bfloat16 *hi = Hc + static_cast<size_t>(r) * d;
            __nv_bfloat16 *lo = Hc_lo ? Hc_lo + static_cast<size_t>(r) * d : nullptr;
            for (int g = threadIdx.x; g < groups; g += blockDim.x)
                gather8(src + 8 * g, hi + 8 * g, lo ? lo + 8 * g : nullptr, live);
        } else if (!live && threadIdx.x == 0) {
            idx[r] = idx[0];
        }
        if (threadIdx.x == 0) {
            const int64_t tt = live ? t[src_row] : -1;
            tc[r] = (tt >= 0 && tt < V) ? static_cast<int>(tt) : -1;
            z[r] = __int_as_float(0x7fc00000);
        }
    }
}

// W (fp32) -> W_hi, W_lo (bf16) for the split-precision path; n % 8 == 0.
__global__ void __launch_bounds__(256)
    k_split_rows(const float *__restrict__ W, size_t n, __nv_bfloat16 *__restrict__ hi, __nv_bfloat16 *__restrict__ lo) {
    const size_t groups = n / 8;
    for (size_t g = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; g < groups;
         g += static_cast<size_t>(gridDim.x) * blockDim.x)
        gather8(W + 8 * g, hi + 8 * g, lo + 8 * g, true);
}

// Merge the per-range (m, l) partials of each row (log2 units) in fixed range
// order: lse2 = M + log2(sum_s l_s 2^(m_s - M)), then loss_i = lse - z_i.
__global__ void __launch_bounds__(256)
    k_lse_merge(const float2 *__restrict__ part, const int *__restrict__ counters, int n_tiles, int num_pairs,
                const float *__restrict__ z, float *__restrict__ lse2_out, float *__restrict__ loss_rows,
                const int *__restrict__ idx, float *__restrict__ lse_user) {
    const int nv = counters[0];
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= nv) return;
    const int m_blocks = cdiv(nv, kPairM);
    const int splits = lse_splits(m_blocks, n_tiles, num_pairs);
    const size_t stride = static_cast<size_t>(m_blocks) * kPairM;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, part[s * stride + row].x);
    float L = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float2 p = part[s * stride + row];
        L += p.y * exp2f(p.x - M);
    }
    const float lse2 = M + log2f(L);
    const float lse = lse2 * 0.6931471805599453f;
    lse2_out[row] = lse2;
    loss_rows[row] = lse - z[row];
    if (lse_user) lse_user[idx[row]] = lse;
}

// Self-test of the bounded wait every pipeline barrier uses: one thread waits
// on a fresh mbarrier that nothing will ever complete, with a limit of
// `cycles` SM clocks. The wait gives up, raises DEV_TIMEOUT in the status
// word and the kernel returns; *out records 1 if the wait reported failure.
__global__ void k_wait_selftest(long long cycles, int *out) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    const bool done = wait_bar(&bar, 0, &abort_flag, cycles);
    out[0] = done ? 0 : 1;
}

// Backward from a stored lse: lse2[r] = lse_in[idx[r]] / ln 2 for the
// compacted rows (the form the G epilogue uses).
__global__ void __launch_bounds__(256)
    k_lse_from_input(const float *__restrict__ lse_in, const int *__restrict__ idx, const int *__restrict__ counters,
                     float *__restrict__ lse2_out) {
    const int nv = counters[0];
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row < nv) lse2_out[row] = lse_in[idx[row]] * kLog2e;
}

// Sum of loss_i over this call's (or token chunk's) valid rows with a fixed
// summation tree (one CTA, fp64), so the result does not depend on scheduling.
__global__ void __launch_bounds__(1024)
    k_loss_partial(const float *__restrict__ loss_rows, const int *__restrict__ counters, double *__restrict__ out) {
    __shared__ double sh[1024];
    const int nv = counters[0];
    double acc = 0.0;
    for (int i = threadIdx.x; i < nv; i += 1024) acc += static_cast<double>(loss_rows[i]);
    sh[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 512; w > 0; w >>= 1) {
        if (static_cast<int>(threadIdx.x) < w) sh[threadIdx.x] += sh[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[0] = sh[0];
}

// loss = (sum of the partial sums, in order) / Nv. Nv = 0 gives 0/0 = NaN.
__global__ void k_loss_final(const double *__restrict__ partials, int n, const int *__restrict__ nv_norm,
                             float *__restrict__ loss) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += partials[i];
    loss[0] = static_cast<float>(s / static_cast<double>(nv_norm[0]));
}

// Number of valid (non-ignored) targets over all N positions, for the
// normaliser when the rows are processed in token chunks.
__global__ void __launch_bounds__(1024)
    k_count_valid(const int64_t *__restrict__ t, int N, int64_t ignore_index, int *__restrict__ count) {
    __shared__ int sh[32];
    int c = 0;
    for (int i = threadIdx.x; i < N; i += 1024) c += t[i] != ignore_index ? 1 : 0;
    for (int o = 16; o > 0; o >>= 1) c += __shfl_down_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x < 32) {
        c = sh[threadIdx.x];
        for (int o = 16; o > 0; o >>= 1) c += __shfl_down_sync(0xffffffffu, c, o);
        if (threadIdx.x == 0) count[0] = c;
    }
}

__device__ __forceinline__ void store_row_elems(__nv_bfloat16 *dst, const float4 a, const float4 b) {
    uint4 v = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    *reinterpret_cast<uint4 *>(dst) = v;
}
__device__ __forceinline__ void store_row_elems(float *dst, const float4 a, const float4 b) {
    reinterpret_cast<float4 *>(dst)[0] = a;
    reinterpret_cast<float4 *>(dst)[1] = b;
}

// dH[i] = dHacc[inv[i]] rounded to the element type; zero on ignored rows.
template <typename T>
__global__ void __launch_bounds__(256)
    k_dh_scatter(const float *__restrict__ dH_acc, const int *__restrict__ inv, int N, int d, T *__restrict__ dH) {
    const int groups = d / 8;   // d is a multiple of 8 elements for bf16, 4 for fp32 (handled below)
    for (int r = blockIdx.x; r < N; r += gridDim.x) {
        const int c = inv[r];
        T *dst = dH + static_cast<size_t>(r) * d;
        const float *src = dH_acc + static_cast<size_t>(c < 0 ? 0 : c) * d;
        for (int g = threadIdx.x; g < groups; g += blockDim.x) {
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (c >= 0) {
                lo = reinterpret_cast<const float4 *>(src)[2 * g];
                hi = reinterpret_cast<const float4 *>(src)[2 * g + 1];
            }
            store_row_elems(dst + 8 * g, lo, hi);
        }
        for (int j = groups * 8 + threadIdx.x; j < d; j += blockDim.x)
            dst[j] = static_cast<T>(c >= 0 ? src[j] : 0.f);
    }
}

}  // namespace lce
