// Input-embedding lookup that skips padding, and its deterministic gradient:
// the input side of a vocabulary matrix W tied to the output projection.
//
//   forward   E[i, :] = W[t_i, :] for t_i != pad_id, a zero row for padding
//             (the valid mask and the lookup in one kernel, no host sync:
//             "为什么26万词表会卡死16GB显卡", section 2.3 稀疏索引引擎)
//   backward  dW[v, :] (+)= sum of dE[i, :] over positions i with t_i == v,
//             each sum taken in a fixed order (the batch's gradient rows
//             aggregated per token after backward, same page, section 2.2;
//             here without atomics, so the result is reproducible bit for bit)
//
// The backward groups the valid positions by token with a stable LSD radix
// sort spread over up to kEmbMaxSortBlocks CTAs: per pass (9-bit digits, as
// many passes as the bits of V - 1 need), k_emb_hist counts each block's
// digits and k_emb_scatter gives every block its offsets (column sums over
// the blocks before it plus the digit totals before its digit) and places
// its elements stably (within a 1024-element sub-chunk: a warp match gives
// the rank among equal digits, per-warp digit counts give the warp's
// offset; sub-chunks in order). The first pass reads the token ids directly
// and drops padding and out-of-range ids, so no separate compaction runs.
// The sorted list is then cut into fixed 32-element chunks: k_emb_segsum
// sums, per chunk and 512-column slice, each run of equal tokens in order,
// straight into dW when the run is the token's whole segment, else into the
// run's partial row; k_emb_combine (256-column slices) adds the partial rows
// of each segment that spans chunks, in chunk order, into dW. dW is fp32, or
// bf16 with every fp32 row sum rounded once as it is stored.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "lce_gemm.cuh"

namespace lce {

constexpr int kEmbSortThreads = 1024;   // threads per sort block: one element each per sub-chunk
constexpr int kEmbRadixBits = 9;
constexpr int kEmbBuckets = 1 << kEmbRadixBits;
constexpr int kEmbMaxSortBlocks = 64;
constexpr int kEmbSegCols = 256;   // columns per combine block (64 threads x 4)
constexpr int kEmbChunk = 32;      // sorted elements per segment-sum chunk

// Sort geometry for N positions: blocks and the elements each block covers
// (a multiple of the sub-chunk), and the partial rows the chunks may need.
__host__ __device__ inline int emb_sort_blocks(int64_t N) {
    const int64_t b = (N + kEmbSortThreads - 1) / kEmbSortThreads;
    return static_cast<int>(b < kEmbMaxSortBlocks ? (b > 0 ? b : 1) : kEmbMaxSortBlocks);
}
__host__ __device__ inline int64_t emb_sort_span(int64_t N) {
    const int64_t b = emb_sort_blocks(N);
    const int64_t per = (N + b - 1) / b;
    return (per + kEmbSortThreads - 1) / kEmbSortThreads * kEmbSortThreads;
}
__host__ __device__ inline int64_t emb_chunks_max(int64_t N) { return (N + kEmbChunk - 1) / kEmbChunk; }
__host__ __device__ inline int emb_radix_passes(int64_t V) {
    int bits = 1;
    while (bits < 31 && (int64_t(1) << bits) < V) ++bits;
    return (bits + kEmbRadixBits - 1) / kEmbRadixBits;
}

template <typename T>
struct Vec4;   // four consecutive elements
template <>
struct Vec4<__nv_bfloat16> {
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float *x) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = __uint_as_float(u.x << 16), x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16), x[3] = __uint_as_float(u.y & 0xffff0000u);
    }
};
template <>
struct Vec4<float> {
    static __device__ __forceinline__ void load(const float *p, float *x) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
    }
};

// One warp per row, 16-byte vectors (rows are d*sizeof(T) bytes, a multiple
// of 16). A non-padding token outside [0, V) gets a zero row and raises
// DEV_TARGET_RANGE in the status word.
template <typename T>
__global__ void __launch_bounds__(256)
    k_emb_forward(const T *__restrict__ W, const int64_t *__restrict__ t, int64_t pad_id, int N, int d, int64_t V,
                  T *__restrict__ E) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    const int vecs = d * static_cast<int>(sizeof(T)) / 16;
    for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < N; row += warps) {
        const int64_t tok = t[row];
        const bool pad = tok == pad_id;
        const bool live = !pad && tok >= 0 && tok < V;
        if (!pad && !live && lane == 0) atomicOr(&g_status, DEV_TARGET_RANGE);
        const uint4 *src = reinterpret_cast<const uint4 *>(W + (live ? tok : 0) * static_cast<int64_t>(d));
        uint4 *dst = reinterpret_cast<uint4 *>(E + static_cast<int64_t>(row) * d);
        for (int k = lane; k < vecs; k += 32) dst[k] = live ? src[k] : make_uint4(0, 0, 0, 0);
    }
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns
// the prefix of this thread and sets *total. Uses warp_incl[32].
__device__ __forceinline__ int block_scan_1024(int x, int *warp_incl, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_incl[warp] = incl;
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
    const int pre = (warp ? warp_incl[warp - 1] : 0) + incl - x;
    *total = warp_incl[31];
    __syncthreads();
    return pre;
}

// One element of a sort pass: pass 0 reads position i of the token ids
// (valid: not padding and inside [0, V)), later passes element i of the
// previous pass's output.
struct EmbSortIn {
    const int64_t *t;    // pass 0: token ids [N]
    const int *keys;     // later passes: sorted keys and positions
    const int *vals;
    int64_t pad_id, V;
    int first;           // 1 on pass 0
    int n;               // pass 0: N; later: read from counts[0]
};
__device__ __forceinline__ bool emb_elem(const EmbSortIn &in, int i, int &key, int &val, bool &bad) {
    bad = false;
    if (in.first) {
        const int64_t tok = in.t[i];
        if (tok == in.pad_id) return false;
        if (tok < 0 || tok >= in.V) {
            bad = true;
            return false;
        }
        key = static_cast<int>(tok);
        val = i;
        return true;
    }
    key = in.keys[i];
    val = in.vals[i];
    return true;
}

// Per block: digit counts of its elements -> hist[digit * blocks + block].
__global__ void __launch_bounds__(kEmbSortThreads)
    k_emb_hist(EmbSortIn in, const int *__restrict__ counts, int span, int shift, int *__restrict__ hist) {
    __shared__ int cnt[kEmbBuckets];
    __shared__ int bad_any;
    const int tid = threadIdx.x;
    for (int b = tid; b < kEmbBuckets; b += kEmbSortThreads) cnt[b] = 0;
    if (tid == 0) bad_any = 0;
    __syncthreads();
    const int n = in.first ? in.n : counts[0];
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * span;
    const int64_t r1 = r0 + span < n ? r0 + span : n;
    bool bad_seen = false;
    for (int64_t i = r0 + tid; i < r1; i += kEmbSortThreads) {
        int key, val;
        bool bad;
        if (emb_elem(in, static_cast<int>(i), key, val, bad)) atomicAdd(&cnt[(key >> shift) & (kEmbBuckets - 1)], 1);
        bad_seen |= bad;
    }
    if (bad_seen) bad_any = 1;
    __syncthreads();
    for (int b = tid; b < kEmbBuckets; b += kEmbSortThreads) hist[b * gridDim.x + blockIdx.x] = cnt[b];
    if (tid == 0 && bad_any) atomicOr(&g_status, DEV_TARGET_RANGE);
}

// Per block: its offsets from the histograms, then a stable placement of its
// elements (sub-chunks of 1024 in order). Block 0 of pass 0 writes the
// number of valid positions to counts[0].
__global__ void __launch_bounds__(kEmbSortThreads)
    k_emb_scatter(EmbSortIn in, int *__restrict__ counts, int span, int shift, const int *__restrict__ hist,
                  int *__restrict__ k_out, int *__restrict__ v_out) {
    __shared__ uint16_t wcnt[32][kEmbBuckets];   // per-warp digit counts, then per-warp offsets
    __shared__ int base[kEmbBuckets];
    __shared__ int ctot[kEmbBuckets];
    __shared__ int warp_incl[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int nb = gridDim.x, b = blockIdx.x;

    // offsets: digit totals before this digit + this digit's count in earlier blocks
    int before = 0, tot = 0;
    if (tid < kEmbBuckets) {
        const int *h = hist + tid * nb;
        for (int j = 0; j < nb; ++j) {
            const int c = h[j];
            tot += c;
            before += j < b ? c : 0;
        }
    }
    int all;
    const int pre = block_scan_1024(tid < kEmbBuckets ? tot : 0, warp_incl, &all);
    if (tid < kEmbBuckets) base[tid] = pre + before;
    if (in.first && b == 0 && tid == 0) counts[0] = all;
    __syncthreads();

    const int n = in.first ? in.n : counts[0];
    const int64_t r0 = static_cast<int64_t>(b) * span;
    const int64_t r1 = r0 + span < n ? r0 + span : n;
    for (int64_t c0 = r0; c0 < r1; c0 += kEmbSortThreads) {
        for (int j = tid; j < 32 * kEmbBuckets / 2; j += kEmbSortThreads) reinterpret_cast<uint32_t *>(&wcnt[0][0])[j] = 0;
        __syncthreads();
        const int64_t i = c0 + tid;
        int key = 0, val = 0;
        bool bad = false;
        const bool live = i < r1 && emb_elem(in, static_cast<int>(i), key, val, bad);
        const int dg = live ? (key >> shift) & (kEmbBuckets - 1) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, dg);
        const int rank = __popc(peers & lt);
        if (live && rank == 0) wcnt[warp][dg] = static_cast<uint16_t>(__popc(peers));
        __syncthreads();
        if (tid < kEmbBuckets) {   // exclusive prefix over warps
            int run = 0;
            for (int w = 0; w < 32; ++w) {
                const int c = wcnt[w][tid];
                wcnt[w][tid] = static_cast<uint16_t>(run);
                run += c;
            }
            ctot[tid] = run;
        }
        __syncthreads();
        if (live) {
            const int dst = base[dg] + wcnt[warp][dg] + rank;
            k_out[dst] = key;
            v_out[dst] = val;
        }
        __syncthreads();
        if (tid < kEmbBuckets) base[tid] += ctot[tid];
        __syncthreads();
    }
}

// Run of equal keys containing sorted index j within [lo, hi): its first index.
__device__ __forceinline__ int emb_run_start(const int *keys, int j, int lo) {
    const int key = keys[j];
    while (j > lo && keys[j - 1] == key) --j;
    return j;
}

// Per (32-element chunk, 512-column slice): the sum of each run of equal
// tokens in order, eight columns per thread (one 16-byte load per bf16 row).
// The chunk's rows are loaded four at a time whatever the run boundaries
// (short runs are the common case), together with dW's current value for
// every run that starts among them (when accumulating), so that a batch
// costs one round trip to memory. A run that is its token's whole segment
// goes into dW; the first / last run of the chunk, when its segment continues
// into the chunk before / after, into partial row 2c / 2c + 1.
constexpr int kEmbRowsInFlight = 4;
constexpr int kEmbSegSumCols = 512;   // columns per segment-sum block (64 threads x 8)

// Eight columns of a dW or partial row: fp32, or bf16 rounded to nearest
// from the fp32 sum (then written once, never accumulated into).
__device__ __forceinline__ void emb_store8(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void emb_store8(__nv_bfloat16 *p, const float *v) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
    *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(h);
}
__device__ __forceinline__ void emb_load8(const __nv_bfloat16 *p, float *x) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) x[2 * k] = __uint_as_float(w[k] << 16), x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
}
__device__ __forceinline__ void emb_load8(const float *p, float *x) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w, x[4] = b.x, x[5] = b.y, x[6] = b.z, x[7] = b.w;
}

template <typename O>
__device__ __forceinline__ void emb_flush(const int *keys, int nv, int c, int j0, int j1, int r0, int r1, int key,
                                          float *acc, const float *wcur, int d, int col, O *dW, float *partial,
                                          int accumulate) {
    const bool before = r0 == j0 && j0 > 0 && keys[j0 - 1] == key;
    const bool after = r1 == j1 && j1 < nv && keys[j1] == key;
    if (!before && !after) {
        if (accumulate) {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += wcur[k];
        }
        emb_store8(dW + static_cast<int64_t>(key) * d + col, acc);
    } else {
        emb_store8(partial + static_cast<int64_t>(2 * c + (r0 == j0 ? 0 : 1)) * d + col, acc);
    }
}

template <typename T, typename O>
__global__ void __launch_bounds__(64, 8)
    k_emb_segsum(const T *__restrict__ dE, const int *__restrict__ counts, const int *__restrict__ keys,
                 const int *__restrict__ order, int d, O *__restrict__ dW, float *__restrict__ partial,
                 int accumulate) {
    const int nv = counts[0];
    const int nchunks = (nv + kEmbChunk - 1) / kEmbChunk;
    const int col = blockIdx.y * kEmbSegSumCols + threadIdx.x * 8;   // d % 8 == 0: all eight inside d
    if (col >= d) return;
    for (int c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int j0 = c * kEmbChunk;
        const int j1 = j0 + kEmbChunk < nv ? j0 + kEmbChunk : nv;
        int key = -1, r0 = j0;
        float wcur[8], acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) wcur[k] = acc[k] = 0.f;
        for (int jb = j0; jb < j1; jb += kEmbRowsInFlight) {
            float x[kEmbRowsInFlight][8], pre[kEmbRowsInFlight][8];
            int kk[kEmbRowsInFlight];
#pragma unroll
            for (int r = 0; r < kEmbRowsInFlight; ++r) kk[r] = jb + r < j1 ? keys[jb + r] : -1;
#pragma unroll
            for (int r = 0; r < kEmbRowsInFlight; ++r) {
                const int j = jb + r;
                const bool starts = j < j1 && kk[r] != (r ? kk[r - 1] : key);
                if (accumulate && starts) {
                    emb_load8(reinterpret_cast<const float *>(dW) + static_cast<int64_t>(kk[r]) * d + col, pre[r]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) pre[r][k] = 0.f;
                }
                if (j < j1) {
                    emb_load8(dE + static_cast<int64_t>(order[j]) * d + col, x[r]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) x[r][k] = 0.f;
                }
            }
#pragma unroll
            for (int r = 0; r < kEmbRowsInFlight; ++r) {
                const int j = jb + r;
                if (j >= j1) break;
                if (kk[r] != key) {   // a run starts here; the one before (if any) is complete
                    if (j > j0) emb_flush(keys, nv, c, j0, j1, r0, j, key, acc, wcur, d, col, dW, partial, accumulate);
#pragma unroll
                    for (int k = 0; k < 8; ++k) acc[k] = 0.f, wcur[k] = pre[r][k];
                    r0 = j;
                    key = kk[r];
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) acc[k] += x[r][k];
            }
        }
        emb_flush(keys, nv, c, j0, j1, r0, j1, key, acc, wcur, d, col, dW, partial, accumulate);
    }
}

// Four columns of a dW row (see emb_store8).
__device__ __forceinline__ void emb_store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void emb_store4(__nv_bfloat16 *p, float4 v) {
    reinterpret_cast<__nv_bfloat162 *>(p)[0] = __floats2bfloat162_rn(v.x, v.y);
    reinterpret_cast<__nv_bfloat162 *>(p)[1] = __floats2bfloat162_rn(v.z, v.w);
}

// Segments that span chunks: the chunk holding a segment's first run adds
// that run's partial row and the following chunks' partial rows of the
// segment, in chunk order, into dW[token]. The block's 64 threads test 64
// chunk boundaries at once to find how far the segment reaches, then each
// thread loads its columns of those partial rows with eight loads in flight.
template <typename O>
__global__ void __launch_bounds__(64, 8)
    k_emb_combine(const int *__restrict__ counts, const int *__restrict__ keys, int d, O *__restrict__ dW,
                  const float *__restrict__ partial, int accumulate) {
    const int nv = counts[0];
    const int nchunks = (nv + kEmbChunk - 1) / kEmbChunk;
    const int col = blockIdx.y * kEmbSegCols + threadIdx.x * 4;
    const bool active = col < d;   // every thread takes part in the block-wide counts below
    for (int c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int j0 = c * kEmbChunk;
        const int j1 = j0 + kEmbChunk < nv ? j0 + kEmbChunk : nv;
        const int key = keys[j1 - 1];
        if (!(j1 < nv && keys[j1] == key)) continue;           // the last run ends in this chunk (uniform)
        const int rs = emb_run_start(keys, j1 - 1, j0);
        if (rs == j0 && j0 > 0 && keys[j0 - 1] == key) continue;   // not the segment's first chunk (uniform)
        // chunks c+1 .. c+len hold the rest of the segment
        int len = 0;
        for (;;) {
            const int64_t e = static_cast<int64_t>(c + len + 1 + threadIdx.x) * kEmbChunk;
            const bool in_seg = e < nv && keys[e] == key;
            const int n = __syncthreads_count(in_seg);
            len += n;
            if (n < static_cast<int>(blockDim.x)) break;
        }
        if (!active) continue;
        O *out = dW + static_cast<int64_t>(key) * d + col;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (accumulate) {   // fp32 dW only
            const float4 a = *reinterpret_cast<const float4 *>(out);
            acc[0] = a.x, acc[1] = a.y, acc[2] = a.z, acc[3] = a.w;
        }
        // partial rows in chunk order: the first chunk's last run, then each
        // following chunk's first run
        for (int q0 = 0; q0 <= len; q0 += 8) {
            float4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int qq = q0 + q;
                const int slot = qq == 0 ? 2 * c + (rs == j0 ? 0 : 1) : 2 * (c + qq);
                v[q] = qq <= len ? *reinterpret_cast<const float4 *>(partial + static_cast<int64_t>(slot) * d + col)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (q0 + q <= len) acc[0] += v[q].x, acc[1] += v[q].y, acc[2] += v[q].z, acc[3] += v[q].w;
        }
        emb_store4(out, make_float4(acc[0], acc[1], acc[2], acc[3]));
    }
}

// dW = 0 (n floats, n % 4 == 0)
__global__ void __launch_bounds__(256) k_zero_f32(float *__restrict__ p, size_t n) {
    const size_t n4 = n / 4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        reinterpret_cast<float4 *>(p)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace lce
