// Input-embedding lookup that skips padding, and its deterministic gradient:
// the input side of a vocabulary matrix W tied to the output projection.
//
//   forward   E[i, :] = W[t_i, :] for t_i != pad_id, a zero row for padding
//             (the valid mask and the lookup in one kernel, no host sync:
//             "为什么26万词表会卡死16GB显卡", section 2.3 稀疏索引引擎)
//   backward  dW[v, :] (+)= sum of dE[i, :] over positions i with t_i == v,
//             each sum taken in ascending position order (the batch's
//             gradient rows aggregated per token after backward, same page,
//             section 2.2; here in a fixed order instead of atomics, so the
//             result is reproducible bit for bit)
//
// The backward groups the valid positions by token with one CTA: compaction
// into (token, position) pairs, then a stable LSD radix sort on the token
// (8-bit digits; within a 1024-element chunk an element's rank among equal
// digits comes from a warp match plus per-warp digit offsets, chunks in
// order), then the list of segment heads (first position of each token).
// Segments are cut into pieces of at most kEmbPiece rows (fixed boundaries,
// so the result does not depend on scheduling). A second kernel sums each
// piece's rows in order, a block per (piece, 256-column slice): a segment of
// one piece goes straight into dW, the pieces of a longer segment into fp32
// partial rows, which a third kernel adds into dW in piece order.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "lce_gemm.cuh"

namespace lce {

constexpr int kEmbSortThreads = 1024;
constexpr int kEmbRadixBits = 8;
constexpr int kEmbBuckets = 1 << kEmbRadixBits;
constexpr int kEmbSegCols = 256;   // columns per segment-sum block (64 threads x 4)
constexpr int kEmbPiece = 64;      // rows per piece of a segment

// Bound on the pieces of N positions and on the partial rows they need.
__host__ __device__ inline int64_t emb_pieces_max(int64_t N) { return N + N / kEmbPiece + 1; }
__host__ __device__ inline int64_t emb_slots_max(int64_t N) { return 2 * (N / kEmbPiece) + 2; }

// Grouping output, in the workspace (filled by k_emb_sort).
struct EmbGroups {
    int *counts;       // [0] valid positions, [1] segments, [2] pieces, [3] multi-piece segments
    int **keys;        // -> token of each sorted position
    int **order;       // -> sorted positions
    int *seg;          // [nseg + 1] first sorted index of each segment
    int *piece_start;  // [npieces] first sorted index of the piece
    int *piece_seg;    // [npieces] its segment
    int *piece_slot;   // [npieces] partial row, or -1 (single-piece segment: straight into dW)
    int *multi_seg;    // [nmulti] segments of more than one piece
    int *multi_slot;   // [nmulti] their first partial row (pieces in order)
    int *multi_np;     // [nmulti] their piece counts
};

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

// Single CTA: valid positions grouped by token, ascending positions within a
// token. Workspace arrays of N int32 each: keys/vals (ping-pong x2), seg
// (N + 1). Out: counts[0] = number of valid positions, counts[1] = number of
// segments; order = the sorted positions, skey = their tokens, seg[s] = first
// index of segment s in order (seg[nseg] = count).
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

__global__ void __launch_bounds__(kEmbSortThreads)
    k_emb_sort(const int64_t *__restrict__ t, int N, int64_t pad_id, int64_t V, int *kA, int *vA, int *kB, int *vB,
               EmbGroups g) {
    int *seg = g.seg;
    int *counts = g.counts;
    __shared__ int wcnt[32][kEmbBuckets];   // per-warp digit counts, then per-warp digit offsets
    __shared__ int base[kEmbBuckets];
    __shared__ int ctot[kEmbBuckets];
    __shared__ int warp_incl[32];
    __shared__ int bad_total;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    if (tid == 0) bad_total = 0;

    // 1. compaction: (token, position) of the valid positions, ascending
    int running = 0, bad = 0;
    for (int b0 = 0; b0 < N; b0 += kEmbSortThreads) {
        const int i = b0 + tid;
        const int64_t tok = i < N ? t[i] : pad_id;
        const bool valid = tok != pad_id && tok >= 0 && tok < V;
        bad += (i < N && tok != pad_id && !valid) ? 1 : 0;
        const unsigned m = __ballot_sync(0xffffffffu, valid);
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
        if (valid) {
            const int pos = running + (warp ? warp_incl[warp - 1] : 0) + __popc(m & lt);
            kA[pos] = static_cast<int>(tok);
            vA[pos] = i;
        }
        running += warp_incl[31];
        __syncthreads();
    }
    if (bad) atomicAdd(&bad_total, bad);
    const int nv = running;

    // 2. stable LSD radix sort on the token
    int bits = 1;
    while (bits < 31 && (int64_t(1) << bits) < V) ++bits;
    int *ks = kA, *vs = vA, *kd = kB, *vd = vB;
    for (int shift = 0; shift < bits; shift += kEmbRadixBits) {
        for (int b = tid; b < kEmbBuckets; b += kEmbSortThreads) base[b] = 0;
        __syncthreads();
        for (int i = tid; i < nv; i += kEmbSortThreads) atomicAdd(&base[(ks[i] >> shift) & (kEmbBuckets - 1)], 1);
        __syncthreads();
        if (warp == 0) {   // exclusive scan of the 256 bucket counts, 8 per lane
            int c[kEmbBuckets / 32], sum = 0;
#pragma unroll
            for (int j = 0; j < kEmbBuckets / 32; ++j) {
                c[j] = base[lane * (kEmbBuckets / 32) + j];
                sum += c[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            int run = incl - sum;
#pragma unroll
            for (int j = 0; j < kEmbBuckets / 32; ++j) {
                base[lane * (kEmbBuckets / 32) + j] = run;
                run += c[j];
            }
        }
        __syncthreads();
        for (int b0 = 0; b0 < nv; b0 += kEmbSortThreads) {
            for (int j = tid; j < 32 * kEmbBuckets; j += kEmbSortThreads) (&wcnt[0][0])[j] = 0;
            __syncthreads();
            const int i = b0 + tid;
            const bool in = i < nv;
            const int key = in ? ks[i] : 0;
            const int val = in ? vs[i] : 0;
            const int dg = in ? (key >> shift) & (kEmbBuckets - 1) : -1;
            const unsigned peers = __match_any_sync(0xffffffffu, dg);
            const int rank = __popc(peers & lt);
            if (in && rank == 0) wcnt[warp][dg] = __popc(peers);
            __syncthreads();
            for (int b = tid; b < kEmbBuckets; b += kEmbSortThreads) {   // exclusive prefix over warps
                int run = 0;
                for (int w = 0; w < 32; ++w) {
                    const int c = wcnt[w][b];
                    wcnt[w][b] = run;
                    run += c;
                }
                ctot[b] = run;
            }
            __syncthreads();
            if (in) {
                const int dst = base[dg] + wcnt[warp][dg] + rank;
                kd[dst] = key;
                vd[dst] = val;
            }
            __syncthreads();
            for (int b = tid; b < kEmbBuckets; b += kEmbSortThreads) base[b] += ctot[b];
            __syncthreads();
        }
        int *tk = ks, *tv = vs;
        ks = kd, vs = vd, kd = tk, vd = tv;
    }

    // 3. segment heads (first index of each token's run), ascending
    int nseg = 0;
    for (int b0 = 0; b0 < nv; b0 += kEmbSortThreads) {
        const int i = b0 + tid;
        const bool head = i < nv && (i == 0 || ks[i] != ks[i - 1]);
        const unsigned m = __ballot_sync(0xffffffffu, head);
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
        if (head) seg[nseg + (warp ? warp_incl[warp - 1] : 0) + __popc(m & lt)] = i;
        nseg += warp_incl[31];
        __syncthreads();
    }
    if (tid == 0) seg[nseg] = nv;
    __syncthreads();

    // 4. pieces of at most kEmbPiece rows; segments of several pieces get
    //    consecutive partial rows and an entry in the multi-piece list
    int npieces = 0, nslots = 0, nmulti = 0;
    for (int b0 = 0; b0 < nseg; b0 += kEmbSortThreads) {
        const int sidx = b0 + tid;
        const int len = sidx < nseg ? seg[sidx + 1] - seg[sidx] : 0;
        const int np = (len + kEmbPiece - 1) / kEmbPiece;
        const int multi = np > 1 ? 1 : 0;
        int tot_p, tot_s, tot_m;
        const int poff = npieces + block_scan_1024(np, warp_incl, &tot_p);
        const int soff = nslots + block_scan_1024(multi ? np : 0, warp_incl, &tot_s);
        const int moff = nmulti + block_scan_1024(multi, warp_incl, &tot_m);
        for (int k = 0; k < np; ++k) {
            g.piece_start[poff + k] = seg[sidx] + k * kEmbPiece;
            g.piece_seg[poff + k] = sidx;
            g.piece_slot[poff + k] = multi ? soff + k : -1;
        }
        if (multi) {
            g.multi_seg[moff] = sidx;
            g.multi_slot[moff] = soff;
            g.multi_np[moff] = np;
        }
        npieces += tot_p;
        nslots += tot_s;
        nmulti += tot_m;
    }
    if (tid == 0) {
        counts[0] = nv;
        counts[1] = nseg;
        counts[2] = npieces;
        counts[3] = nmulti;
        g.keys[0] = ks;
        g.order[0] = vs;
        if (bad_total) atomicOr(&g_status, DEV_TARGET_RANGE);
    }
}

// Sum of one piece's rows in order, four columns per thread, sixteen rows
// in flight: into dW (single-piece segment; added to dW's value when
// accumulating) or into the piece's partial row. A block per (piece,
// 256-column slice).
constexpr int kEmbRowsInFlight = 16;
template <typename T>
__global__ void __launch_bounds__(64, 8)
    k_emb_pieces(const T *__restrict__ dE, EmbGroups g, int d, float *__restrict__ dW, float *__restrict__ partial,
                 int accumulate) {
    const int npieces = g.counts[2];
    const int *keys = g.keys[0];
    const int *order = g.order[0];
    const int col = blockIdx.y * kEmbSegCols + threadIdx.x * 4;
    if (col >= d) return;
    for (int p = blockIdx.x; p < npieces; p += gridDim.x) {
        const int sidx = g.piece_seg[p];
        const int j0 = g.piece_start[p];
        const int send = g.seg[sidx + 1];
        const int j1 = j0 + kEmbPiece < send ? j0 + kEmbPiece : send;
        const int slot = g.piece_slot[p];
        float *out = slot < 0 ? dW + static_cast<int64_t>(keys[j0]) * d + col : partial + static_cast<int64_t>(slot) * d + col;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (slot < 0 && accumulate) {
            const float4 a = *reinterpret_cast<const float4 *>(out);
            acc[0] = a.x, acc[1] = a.y, acc[2] = a.z, acc[3] = a.w;
        }
        int j = j0;
        for (; j + kEmbRowsInFlight <= j1; j += kEmbRowsInFlight) {
            float x[kEmbRowsInFlight][4];
#pragma unroll
            for (int r = 0; r < kEmbRowsInFlight; ++r)
                Vec4<T>::load(dE + static_cast<int64_t>(order[j + r]) * d + col, x[r]);
#pragma unroll
            for (int r = 0; r < kEmbRowsInFlight; ++r)
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] += x[r][k];
        }
        for (; j < j1; ++j) {
            float x[4];
            Vec4<T>::load(dE + static_cast<int64_t>(order[j]) * d + col, x);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] += x[k];
        }
        *reinterpret_cast<float4 *>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
}

// dW[v] (+)= the partial rows of a multi-piece segment, in piece order.
__global__ void __launch_bounds__(64, 8)
    k_emb_combine(EmbGroups g, int d, float *__restrict__ dW, const float *__restrict__ partial, int accumulate) {
    const int nmulti = g.counts[3];
    const int *keys = g.keys[0];
    const int col = blockIdx.y * kEmbSegCols + threadIdx.x * 4;
    if (col >= d) return;
    for (int m = blockIdx.x; m < nmulti; m += gridDim.x) {
        float *out = dW + static_cast<int64_t>(keys[g.seg[g.multi_seg[m]]]) * d + col;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (accumulate) {
            const float4 a = *reinterpret_cast<const float4 *>(out);
            acc[0] = a.x, acc[1] = a.y, acc[2] = a.z, acc[3] = a.w;
        }
        const float *src = partial + static_cast<int64_t>(g.multi_slot[m]) * d + col;
        for (int k = 0; k < g.multi_np[m]; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(src + static_cast<int64_t>(k) * d);
            acc[0] += a.x, acc[1] += a.y, acc[2] += a.z, acc[3] += a.w;
        }
        *reinterpret_cast<float4 *>(out) = make_float4(acc[0], acc[1], acc[2], acc[3]);
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
