// Persistent, warp-specialised tcgen05 GEMM engine with the fused epilogues
// of the output-projection + cross-entropy path.
//
// One CTA per SM; CTA pairs (clusters of 2) share each 256x256 tile; 192
// threads per CTA:
//   warp 0      TMA producer: streams this CTA's 128 A rows and 128 of the
//               256 B rows per k-block into a 6-stage shared-memory ring
//               (5 stages in the fused-optimizer instantiation; 128-byte
//               swizzle); both CTAs signal the even CTA's barrier.
//   warp 1      allocates TMEM (512 columns = two 128x256 fp32 accumulators
//               per CTA); on the even CTA one thread issues
//               tcgen05.mma.cta_group::2.kind::f16 256x256x16 (bf16 in, fp32
//               accumulate) reading both CTAs' shared memory.
//   warps 2..5  epilogue: tcgen05.ld the finished accumulator (warp w reads
//               TMEM lanes 32*(w%4)..+31, one tile row per thread) while the
//               MMA thread already fills the other accumulator.
//
// Tile types (D = A . B^T in TMEM):
//   T_LSE  S = Hc . W^T       per 256-row pair block over a contiguous range
//          of 256-wide vocab tiles; the epilogue carries the online (max, sum)
//          of exp over the row in registers and writes one (m, l) partial per
//          row and range, plus the target logit (forward).
//   T_G    S = Hc . W_c^T     over one vocab chunk (logits recomputed in
//          backward); the epilogue forms G = (exp(S - lse) - onehot) * scale/Nv
//          and stores it (bf16).
//   T_DW   dW_c = G^T . Hc    (M = chunk vocab rows, K = valid tokens); A and
//          B are read MN-major straight from G and Hc. With a fused optimizer
//          (KIND_BWD_OPT) the epilogue applies the SGD / AdamW update to those
//          W rows instead of storing dW (no dW buffer exists): the TMA engine
//          streams boxes of the rows' weights and optimizer state through a
//          ring in the warp's staging area, each lane updates its row from
//          its TMEM gradient, and the boxes are stored back.
//   T_DH   dHacc (+)= G . W_c (M = valid tokens, K = chunk vocab rows); B is
//          read MN-major straight from W.
//
// Row gather (optional; bf16 inputs, d a multiple of 256): instead of a
// compacted copy Hc, the producer warp loads the valid rows of H itself, each
// lane one tile::gather4 of four rows x 128 bytes per stage (32 lanes: the 128
// rows of a K-major A block, or 64 token rows x 2 column blocks of an MN-major
// B), with row numbers from the compaction index.
//
// Split precision (fp32 inputs): every fp32 operand x is carried as two bf16
// tensors, x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), and the K loop
// runs three segments, A_hi.B_hi + A_hi.B_lo + A_lo.B_hi, into the same
// accumulator (the lo.lo term is below fp32 resolution of the sum). With
// nseg = 1 only the hi tensors are read.
//
// Every wait is bounded: on time-out the CTA raises LCE_DEV_TIMEOUT in the
// device status word, lets its in-flight copies and MMAs land, frees TMEM and
// returns.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "tc_ptx.cuh"

namespace lce {

constexpr int kBM = 128;          // tile rows held by one CTA (TMEM lanes)
constexpr int kPairM = 256;       // tile rows of a CTA pair (UMMA M with cta_group::2)
constexpr int kBN = 256;          // tile cols (UMMA N), split 128 + 128 across the pair
constexpr int kHalfN = 128;       // B rows (N) loaded by each CTA of the pair
constexpr int kBK = 64;           // k per stage: one 128-byte bf16 line
constexpr int kUmmaK = 16;        // k per tcgen05.mma (bf16)
constexpr int kAtom = 64;         // MN elements per 128-byte line
constexpr int kAtomBytes = kBK * 128;   // one MN-major box {64 (MN), 64 (K)} = 8 KB
constexpr int kStages = 6;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;    // two 256-column fp32 accumulators
constexpr int kStageA = kBM * 128;      // this CTA's 128 A rows x 64 k
constexpr int kStageB = kHalfN * 128;   // this CTA's 128 B rows x 64 k
constexpr int kStageBytes = kStageA + kStageB;
constexpr int kPairTx = 2 * kStageBytes;   // bytes both CTAs land on the even CTA's full barrier
// Epilogue staging: each of the 4 epilogue warps owns two 4 KB buffers; a
// 32-row x 32-column chunk (fp32, or bf16 hi + lo) is written there in the
// TMA swizzle pattern and stored to global memory by one bulk tensor store.
constexpr int kEpiBufBytes = 4096;
constexpr int kEpiBytes = 4 * 2 * kEpiBufBytes;
constexpr int kBarrierBytes = 320;   // mbarriers, TMEM address slot and abort flag
constexpr int kGemmSmem = kStages * kStageBytes + kEpiBytes + 1024 /*alignment slack*/ + kBarrierBytes;
// The optimizer instantiation runs a 5-stage ring: the freed 32 KB doubles
// each epilogue warp's staging area (16 KB), which holds the ring of W and
// optimizer-state boxes the TMA engine streams through (the mainloop is as
// fast with 5 stages as with 6 on these shapes).
template <int KIND>
struct Cfg {
    static constexpr int kS = KIND == 2 /* KIND_BWD_OPT */ ? 5 : kStages;
    static constexpr int kEpiWarp = (kGemmSmem - kS * kStageBytes - 1024 - kBarrierBytes) / 4;   // staging bytes per warp
};
constexpr int kOptLoadBars = 5;   // TMA load barriers per epilogue warp (optimizer ring)
constexpr long long kWaitCycles = 2000000000LL;   // ~1 s: far above any legitimate wait
constexpr long long kDrainCycles = 200000000LL;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kFmtBf16 = 1u;   // operand format code of bf16 in the f16-kind descriptor

enum DevStatus : int { DEV_TARGET_RANGE = 1, DEV_TIMEOUT = 2 };

// Device status word (LCE_DEV_* bits). The library is one translation unit,
// so this header is the single definition.
__device__ int g_status = 0;

__host__ __device__ inline int cdiv(int a, int b) { return (a + b - 1) / b; }

// Vocab splits for the LSE pass: choose the number of contiguous vocab ranges
// per 256-row block so that m_blocks*splits units fill whole waves of `sms`
// CTA pairs with the shortest longest-pair time,
// ceil(units/sms) * ceil(n_tiles/splits).
__host__ __device__ inline int lse_splits(int m_blocks, int n_tiles, int sms) {
    if (m_blocks <= 0 || n_tiles <= 1) return 1;
    int best = 1;
    long long best_cost = static_cast<long long>(cdiv(m_blocks, sms)) * n_tiles;
    for (int w = 1; w <= 16; ++w) {
        int s = (w * sms) / m_blocks;
        if (s < 1) continue;
        if (s > n_tiles) s = n_tiles;
        long long cost = static_cast<long long>(cdiv(m_blocks * s, sms)) * cdiv(n_tiles, s);
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Largest number of (m, l) partial rows the LSE pass can write for row
// capacity `rows_cap` (a multiple of 256) and `pairs` CTA pairs.
__host__ __device__ inline long long lse_partial_rows(int rows_cap, int pairs) {
    long long a = 16LL * pairs, b = rows_cap / kPairM;
    return (a > b ? a : b) * kPairM;
}

// Tile types. KIND_LSE launches run only T_LSE; a KIND_BWD launch for vocab
// chunk j runs the G tiles of chunk j+1 (into the next of three G buffers)
// and the dW and dH tiles of chunk j, which are independent of one another,
// so a launch needs no synchronisation inside it. Consecutive KIND_BWD
// launches overlap (programmatic dependent launch): a launch's G tiles start
// on the SMs its predecessor frees, and its dW/dH tiles wait for the
// predecessor (which wrote G_j and the dH accumulator) to complete.
// KIND_BWD_OPT is KIND_BWD with an optimizer step fused into the dW
// epilogue: its own instantiation, so the plain backward keeps its register
// allocation.
enum Kind : int { KIND_LSE = 0, KIND_BWD = 1, KIND_BWD_OPT = 2 };
enum TileType : int { T_LSE = 0, T_G = 1, T_DH = 2, T_DW = 3 };

// Operand tensor maps per tile type: slot 0 = LSE / G (A = Hc K-major,
// B = W K-major), slot 1 = DH (A = G K-major, B = W MN-major), slot 2 = DW
// (A = G MN-major, B = Hc MN-major); [0] = hi (bf16) parts, [1] = lo parts.
struct OperandMaps {
    CUtensorMap A[2];
    CUtensorMap B[2];
};
struct GemmMaps {
    OperandMaps t[3];
    // bulk-store maps (box 32 x 32): G chunk being written (hi, lo; bf16,
    // 64-byte swizzle), dW and the dH accumulator (fp32, 128-byte swizzle)
    CUtensorMap st_g[2];
    CUtensorMap st_dw;
    CUtensorMap st_dh;
    // fused optimizer: {16, 32} boxes of W's state (fp32, 64-byte swizzle:
    // first moment / momentum buffer, second moment, fp32 weights or master
    // copy) and of a bf16 W (32-byte swizzle); unused maps stay zero
    CUtensorMap opt_m, opt_v, opt_w32, opt_w16;
};

__host__ __device__ constexpr int map_slot(int type) { return type == T_DH ? 1 : (type == T_DW ? 2 : 0); }

enum OptKind : int { OPT_NONE = 0, OPT_SGD = 1, OPT_ADAMW = 2 };

// Optimizer update fused into the dW epilogue (the gradient of W never
// reaches memory). SGD: g' = g + wd*w; with momentum b = g' on the first step,
// else b = momentum*b + g', and g' = b; w -= lr*g'. AdamW (decoupled decay):
// w *= 1 - lr*wd; m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*g^2;
// w -= step_size * m / (sqrt(v) * inv_bc2_sqrt + eps), with
// step_size = lr / (1 - b1^t) and inv_bc2_sqrt = 1 / sqrt(1 - b2^t).
struct OptArgs {
    int kind;              // OptKind
    int first;             // SGD: this step starts the momentum buffer
    float lr, wd, momentum, beta1, beta2, eps, step_size, inv_bc2_sqrt;
    void *W;               // [V][d] weights updated in place: bf16, or fp32 when w_fp32
    int w_fp32;
    float *master;         // optional fp32 [V][d] master copy of a bf16 W (W = its bf16 rounding)
    void *m, *v;           // [V][d]: AdamW moments / SGD momentum buffer (m), fp32 or bf16
    int s16;               // m and v are bf16 (read, updated in fp32, stored rounded to nearest)
};

struct GemmArgs {
    const int *counters;   // counters[0] = valid rows this launch tiles (written by the compaction kernel)
    const int *nv_norm;    // *nv_norm = Nv of the whole call, the loss normaliser
    int d, V;
    int num_pairs;         // CTA pairs in the grid (gridDim.x / 2)
    int nseg;              // 1 (bf16 operands) or 3 (split-precision fp32 operands)
    const int *tc;         // compacted targets, -1 where none
    // KIND_LSE
    float *z;              // per compacted row: target logit
    float2 *part;          // (m, l) partials [splits][m_blocks*256]
    // KIND_BWD: dH tiles of the current chunk [v0, v0+vlen) (if has_cur),
    // dW tiles of chunk [v0w, v0w+vlenw) (if has_dw: the current chunk, or
    // the previous one when an optimizer update is fused), G tiles of the
    // next chunk [v0n, v0n+vlenn) (if has_next)
    int v0, vlen, v0n, vlenn, has_cur, has_next, v0w, vlenw, has_dw;
    const float *lse2;     // per compacted row: lse / ln 2
    float *dW;             // [V][d] fp32, or bf16 when dw_bf16
    int acc_dw;            // add into dW instead of overwriting
    int dw_bf16;           // dW is written as bf16 (each fp32 accumulator rounded to nearest)
    float *dH_acc;         // [rows][d] fp32
    int acc_dh;            // add into dHacc (every chunk after the first)
    float grad_scale;      // multiplies G
    const float *grad_ptr; // optional device scalar that also multiplies G
    // MN-major operand maps that are 3-D ({64 within a 128-byte line, K rows,
    // 64-wide column blocks}: one box per operand per stage) instead of 2-D
    // (one {64, 64} box per column block); 3-D needs the MN extent to be a
    // multiple of 64. Bit 0: DW's A (G), bit 1: DW's B (Hc), bit 2: DH's B (W).
    int mn3d;
    // Row gather: the Hc operand (A of LSE / G tiles, B of DW tiles) is read
    // straight from the caller's bf16 H through the compaction index, rows
    // idx[r] (padded rows repeat a valid row; their G rows are zero), by
    // tile::gather4 loads; the operand map is then a {64, 1}-box map of H.
    int gather;
    const int *idx;
    OptArgs opt;
};

struct Sched {
    int units;
    // KIND_LSE (row blocks taken in groups of rgroup)
    int m_blocks, n_tiles, splits, kseg, rgroup;
    // KIND_BWD: task counts and shapes per type (tasks listed G, dW, dH)
    int n_dw, n_dh, n_g, nt_d, nt_g, kseg_dw, kseg_dh, kseg_g;
};

// LSE unit u -> (split, row block). Units run split-major: the pairs running
// together read the same W tiles (each W tile once from DRAM) and every row
// block of H. When those row blocks exceed kLseGroupBytes they are taken in
// balanced groups (split-major within a group), so the H blocks that pairs
// re-read per vocab tile stay in L2, at the cost of one pass over W per
// group: for 39 row blocks of d = 4096 (78 MB) this cut the LSE launch's
// DRAM reads by two thirds (3.2 -> 1.1 GB for a 24576-row vocab slice) and
// the step by 4%. A 48 MB budget (two groups for 29 row blocks of d = 4096,
// 58 MB) is 1% faster per step than one group there; three groups (24 MB)
// are slower again, and 69 MB of row blocks of d = 2048 gain nothing.
constexpr long long kLseGroupBytes = 48LL << 20;
__host__ __device__ inline int lse_group_rows(int m_blocks, int d, int nseg) {
    const long long block_bytes = static_cast<long long>(kPairM) * d * 2 * (nseg > 1 ? 2 : 1);
    long long r = kLseGroupBytes / block_bytes;
    if (r < 1) r = 1;
    if (r >= m_blocks) return m_blocks;
    const int ngroups = static_cast<int>((m_blocks + r - 1) / r);
    return (m_blocks + ngroups - 1) / ngroups;   // balanced group size
}
__device__ __forceinline__ void lse_unit(int m_blocks, int splits, int rg, int u, int &split, int &mb) {
    const int full = m_blocks / rg;   // groups of exactly rg row blocks
    if (u < full * rg * splits) {
        const int g = u / (rg * splits), rem = u % (rg * splits);
        split = rem / rg;
        mb = g * rg + rem % rg;
    } else {
        const int u2 = u - full * rg * splits, rl = m_blocks - full * rg;
        split = u2 / rl;
        mb = full * rg + u2 % rl;
    }
}

struct TileInfo {
    int type, mb, nt, kseg;
};

template <int KIND>
__device__ inline Sched make_sched(const GemmArgs &a, int nv) {
    Sched s{};
    if (KIND == KIND_LSE) {
        s.m_blocks = cdiv(nv, kPairM);
        s.n_tiles = cdiv(a.V, kBN);
        s.kseg = cdiv(a.d, kBK);
        s.splits = lse_splits(s.m_blocks, s.n_tiles, a.num_pairs);
        s.rgroup = lse_group_rows(s.m_blocks, a.d, a.nseg);
        s.units = s.m_blocks * s.splits;
    } else {
        s.nt_d = cdiv(a.d, kBN);
        s.nt_g = a.has_next ? cdiv(a.vlenn, kBN) : 0;
        s.n_dw = a.has_dw ? cdiv(a.vlenw, kPairM) * s.nt_d : 0;
        s.n_dh = a.has_cur ? cdiv(nv, kPairM) * s.nt_d : 0;
        s.n_g = a.has_next ? cdiv(nv, kPairM) * s.nt_g : 0;
        s.kseg_dw = cdiv(nv, kBK);
        s.kseg_dh = cdiv(a.vlen, kBK);
        s.kseg_g = cdiv(a.d, kBK);
        s.units = s.n_g + s.n_dw + s.n_dh;
    }
    return s;
}

// Unit u -> [n0, n1) tiles. LSE units are (256-row block, contiguous vocab range),
// split-major so CTAs running together share W tiles in L2; BWD units are one
// tile each: first the G tiles of the next chunk, which do not depend on the
// previous launch and so can run while its last tiles finish, then dW (long K)
// and dH of the current chunk; d / vocab tiles fastest.
template <int KIND>
__device__ inline void unit_range(const Sched &s, int u, int &n0, int &n1) {
    if (KIND == KIND_LSE) {
        int split, mb;
        lse_unit(s.m_blocks, s.splits, s.rgroup, u, split, mb);
        n0 = static_cast<int>(static_cast<long long>(split) * s.n_tiles / s.splits);
        n1 = static_cast<int>(static_cast<long long>(split + 1) * s.n_tiles / s.splits);
    } else {
        n0 = 0;
        n1 = 1;
    }
}

template <int KIND>
__device__ inline TileInfo tile_info(const Sched &s, int u, int n) {
    TileInfo t;
    if (KIND == KIND_LSE) {
        t.type = T_LSE;
        int split;
        lse_unit(s.m_blocks, s.splits, s.rgroup, u, split, t.mb);
        t.nt = n;
        t.kseg = s.kseg;
    } else if (u < s.n_g) {
        t.type = T_G;
        t.mb = u / s.nt_g;
        t.nt = u % s.nt_g;
        t.kseg = s.kseg_g;
    } else if (u < s.n_g + s.n_dw) {
        const int q = u - s.n_g;
        t.type = T_DW;
        t.mb = q / s.nt_d;
        t.nt = q % s.nt_d;
        t.kseg = s.kseg_dw;
    } else {
        const int q = u - s.n_g - s.n_dw;
        t.type = T_DH;
        t.mb = q / s.nt_d;
        t.nt = q % s.nt_d;
        t.kseg = s.kseg_dh;
    }
    return t;
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                         long long limit = kWaitCycles) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(&g_status, DEV_TIMEOUT);
            return false;
        }
    }
}

// Wait used only while shutting down after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    while (!mbar_try_wait(a, parity)) {
        if (clock64() - t0 > kDrainCycles) return;
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// fp32 -> (hi, lo) with hi = bf16(x) and lo = x - hi (exact in fp32; the
// caller rounds lo to bf16 when it stores it).
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    const float h = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - h;
    hi = h;
}

// Fused optimizer step on one 32-row x 16-column box of W held in a warp's
// staging buffer, as the TMA engine loaded it: lane r updates row r from its
// gradient g[0..15] (straight from TMEM). Buffer layout: first moment /
// momentum buffer (fp32, 2 KB, or bf16 in its first 1 KB), second moment
// (likewise), then the weights: fp32 (2 KB; the master copy or an fp32 W) or
// bf16 (1 KB); with a master copy the bf16 rounding of W follows at 6 KB.
// fp32 rows of 64 bytes keep 16-byte unit k of row r at unit k ^ ((r >> 1)
// & 3) (64-byte swizzle), bf16 rows of 32 bytes at unit k ^ ((r >> 2) & 1)
// (32-byte swizzle).
// Byte offsets in one ring buffer: fp32 state {m 0, v 2048, weights 4096,
// bf16 W out 6144}; bf16 state {m 0, v 1024, weights 2048, bf16 W out 4096}.
struct OptLayout {
    int m, v, w, wout;
};
__device__ __forceinline__ OptLayout opt_layout(const OptArgs &o) {
    return o.s16 ? OptLayout{0, 1024, 2048, 4096} : OptLayout{0, 2048, 4096, 6144};
}

__device__ __forceinline__ float4 *opt_f32(uint8_t *buf, int off, int r, int k) {
    return reinterpret_cast<float4 *>(buf + off + r * 64 + ((k ^ ((r >> 1) & 3)) << 4));
}
__device__ __forceinline__ uint4 *opt_b16(uint8_t *buf, int off, int r, int k) {
    return reinterpret_cast<uint4 *>(buf + off + r * 32 + ((k ^ ((r >> 2) & 1)) << 4));
}

// eight bf16 (16 bytes) <-> eight floats
__device__ __forceinline__ void unpack_bf16x8(uint4 x, float *f) {
    const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float *f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

__device__ __forceinline__ void opt_row(const OptArgs &o, uint8_t *buf, int r, const float *g) {
    const bool use_m = o.kind == OPT_ADAMW || o.momentum != 0.f;
    const bool w32 = o.master || o.w_fp32;
    const OptLayout L = opt_layout(o);
    float w[16], m[16], v[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (w32) {
            const float4 x = *opt_f32(buf, L.w, r, k);
            w[4 * k] = x.x, w[4 * k + 1] = x.y, w[4 * k + 2] = x.z, w[4 * k + 3] = x.w;
        }
        if (use_m && !o.s16) {
            const float4 x = *opt_f32(buf, L.m, r, k);
            m[4 * k] = x.x, m[4 * k + 1] = x.y, m[4 * k + 2] = x.z, m[4 * k + 3] = x.w;
        }
        if (o.kind == OPT_ADAMW && !o.s16) {
            const float4 x = *opt_f32(buf, L.v, r, k);
            v[4 * k] = x.x, v[4 * k + 1] = x.y, v[4 * k + 2] = x.z, v[4 * k + 3] = x.w;
        }
    }
    if (o.s16) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (use_m) unpack_bf16x8(*opt_b16(buf, L.m, r, k), m + 8 * k);
            if (o.kind == OPT_ADAMW) unpack_bf16x8(*opt_b16(buf, L.v, r, k), v + 8 * k);
        }
    }
    if (!w32) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 x = *opt_b16(buf, L.w, r, k);
            const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[8 * k + 2 * i] = __uint_as_float(u[i] << 16);
                w[8 * k + 2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (o.kind == OPT_ADAMW) {
            w[j] *= 1.f - o.lr * o.wd;
            m[j] = o.beta1 * m[j] + (1.f - o.beta1) * g[j];
            v[j] = o.beta2 * v[j] + (1.f - o.beta2) * g[j] * g[j];
            w[j] -= o.step_size * m[j] / (sqrtf(v[j]) * o.inv_bc2_sqrt + o.eps);
        } else {
            float dd = g[j] + o.wd * w[j];
            if (use_m) {
                m[j] = o.first ? dd : o.momentum * m[j] + dd;
                dd = m[j];
            }
            w[j] -= o.lr * dd;
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (use_m && !o.s16) *opt_f32(buf, L.m, r, k) = make_float4(m[4 * k], m[4 * k + 1], m[4 * k + 2], m[4 * k + 3]);
        if (o.kind == OPT_ADAMW && !o.s16)
            *opt_f32(buf, L.v, r, k) = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        if (w32) *opt_f32(buf, L.w, r, k) = make_float4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
    if (o.s16) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            if (use_m) *opt_b16(buf, L.m, r, k) = pack_bf16x8(m + 8 * k);
            if (o.kind == OPT_ADAMW) *opt_b16(buf, L.v, r, k) = pack_bf16x8(v + 8 * k);
        }
    }
    if (!o.w_fp32) {
        const int off = o.master ? L.wout : L.w;
#pragma unroll
        for (int k = 0; k < 2; ++k)
            *opt_b16(buf, off, r, k) = make_uint4(pack_bf16x2(w[8 * k], w[8 * k + 1]), pack_bf16x2(w[8 * k + 2], w[8 * k + 3]),
                                                  pack_bf16x2(w[8 * k + 4], w[8 * k + 5]),
                                                  pack_bf16x2(w[8 * k + 6], w[8 * k + 7]));
    }
}

// One warp's ring of optimizer boxes: `nbuf` buffers of `bsz` bytes, one TMA
// load barrier each; box p of a dW tile covers W rows [row, row + 32) and
// columns [col0 + 16p, +16).
struct OptRing {
    uint8_t *base;
    uint64_t *bar;
    int nbuf, bsz;
    uint32_t bytes;    // transaction bytes of one box's loads
    uint32_t phase;    // bit b: parity of buffer b's next completion
    uint32_t pend;     // bit b: a load into buffer b is in flight
};

// lane 0: load box p (state and weights) into its ring buffer
__device__ __forceinline__ void opt_issue(const GemmMaps &maps, const OptArgs &o, OptRing &q, int p, int col,
                                          int row) {
    const int b = p % q.nbuf;
    uint8_t *buf = q.base + b * q.bsz;
    uint64_t *bar = q.bar + b;
    mbar_arrive_expect_tx(bar, q.bytes);
    const OptLayout L = opt_layout(o);
    if (o.kind == OPT_ADAMW || o.momentum != 0.f) tma_load_2d(buf + L.m, &maps.opt_m, bar, col, row);
    if (o.kind == OPT_ADAMW) tma_load_2d(buf + L.v, &maps.opt_v, bar, col, row);
    if (o.master || o.w_fp32)
        tma_load_2d(buf + L.w, &maps.opt_w32, bar, col, row);
    else
        tma_load_2d(buf + L.w, &maps.opt_w16, bar, col, row);
    q.pend |= 1u << b;
}

// lane 0: store box p back (rows past V and columns past d are clipped)
__device__ __forceinline__ void opt_store(const GemmMaps &maps, const OptArgs &o, const OptRing &q, int p, int col,
                                          int row) {
    const uint8_t *buf = q.base + (p % q.nbuf) * q.bsz;
    const OptLayout L = opt_layout(o);
    if (o.kind == OPT_ADAMW || o.momentum != 0.f) tma_store_2d(&maps.opt_m, buf + L.m, col, row);
    if (o.kind == OPT_ADAMW) tma_store_2d(&maps.opt_v, buf + L.v, col, row);
    if (o.master || o.w_fp32) tma_store_2d(&maps.opt_w32, buf + L.w, col, row);
    if (!o.w_fp32) tma_store_2d(&maps.opt_w16, buf + (o.master ? L.wout : L.w), col, row);
    bulk_commit_group();
}

// Issue this CTA's TMA loads of one k-block (A rows am.., B rows bn.., k0..)
// of tile t into stage (sa, sb), completing on the even CTA's barrier fb.
__device__ __forceinline__ void load_operands(const TileInfo &t, const GemmArgs &a, const CUtensorMap *ma,
                                              const CUtensorMap *mbp, uint8_t *sa, uint8_t *sb, uint32_t fb, int am,
                                              int bn, int k0) {
    if (t.type == T_LSE || t.type == T_G) {
        const int vb = (t.type == T_G ? a.v0n : 0) + bn;
        tma_load_2d_pair(sa, ma, fb, k0, am);
        tma_load_2d_pair(sb, mbp, fb, k0, vb);
    } else if (t.type == T_DH) {
        tma_load_2d_pair(sa, ma, fb, k0, am);
        if (a.mn3d & 4) {
            tma_load_3d_pair(sb, mbp, fb, 0, a.v0 + k0, bn / kAtom);
        } else {
#pragma unroll
            for (int b = 0; b < kHalfN / kAtom; ++b)
                tma_load_2d_pair(sb + b * kAtomBytes, mbp, fb, bn + b * kAtom, a.v0 + k0);
        }
    } else {
        if (a.mn3d & 1) {
            tma_load_3d_pair(sa, ma, fb, 0, k0, am / kAtom);
        } else {
#pragma unroll
            for (int b = 0; b < kBM / kAtom; ++b) tma_load_2d_pair(sa + b * kAtomBytes, ma, fb, am + b * kAtom, k0);
        }
        if (a.mn3d & 2) {
            tma_load_3d_pair(sb, mbp, fb, 0, k0, bn / kAtom);
        } else {
#pragma unroll
            for (int b = 0; b < kHalfN / kAtom; ++b)
                tma_load_2d_pair(sb + b * kAtomBytes, mbp, fb, bn + b * kAtom, k0);
        }
    }
}

// TMA producer of one CTA: waits for free stages and issues this CTA's loads
// of every k-block of its tiles, completing on the even CTA's full barrier.
// kGather = false runs on one thread (lane 0): the producer's reaction time
// per stage is on the MMA's critical path, so no warp-wide step is taken.
// kGather = true runs on the whole warp: lane 0 waits and issues the tiled
// loads, and every lane issues one tile::gather4 of the gathered operand.
template <int KIND, bool kGather>
__device__ __forceinline__ void producer(const GemmMaps &maps, const GemmArgs &a, const Sched &s, int pair,
                                         int npairs, uint32_t rank, int lane, uint8_t *smem, uint64_t *full,
                                         uint64_t *empty, uint32_t full_even, volatile int *abort_flag) {
    constexpr int S = Cfg<KIND>::kS;
    int it = 0;
    bool ok = true;
    bool dep_done = false;
    const int arow = static_cast<int>(rank) * kBM;      // this CTA's A rows within the pair tile
    const int brow = static_cast<int>(rank) * kHalfN;   // this CTA's B rows (N) within the tile
    const int4 *idx4 = reinterpret_cast<const int4 *>(a.idx);
    for (int u = pair; ok && u < s.units; u += npairs) {
        int n0, n1;
        unit_range<KIND>(s, u, n0, n1);
        for (int n = n0; ok && n < n1; ++n) {
            const TileInfo t = tile_info<KIND>(s, u, n);
            if (KIND != KIND_LSE && !dep_done && t.type != T_G) {
                // dW / dH read what the previous launch wrote; every thread
                // that issues loads waits
                griddep_wait();
                if (lane == 0) griddep_launch_dependents();
                dep_done = true;
            }
            const OperandMaps &om = maps.t[map_slot(t.type)];
            const int k_blocks = t.kseg * a.nseg;
            const int am = t.mb * kPairM + arow;   // first A row (M) of this CTA
            const int bn = t.nt * kBN + brow;      // first B row (N) of this CTA
            const bool gA = kGather && (t.type == T_LSE || t.type == T_G);
            const bool gB = kGather && t.type == T_DW;
            int4 rows = make_int4(0, 0, 0, 0);     // this lane's four gathered rows
            if (gA) rows = idx4[(am >> 2) + lane];
            int4 rows_next = rows;
            if (gB && k_blocks > 0) rows_next = idx4[(lane & 15)];
            for (int kbt = 0; kbt < k_blocks; ++kbt, ++it) {
                const int st = it % S;
                if (gB) {
                    // token rows of this k-block; the next block's are fetched
                    // before the wait so that their latency overlaps it
                    rows = rows_next;
                    if (kbt + 1 < k_blocks) rows_next = idx4[(((kbt + 1) * kBK) >> 2) + (lane & 15)];
                }
                if (kGather) {
                    bool got = true;
                    if (lane == 0) got = wait_bar(&empty[st], ((it / S) & 1) ^ 1, abort_flag);
                    if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
                        ok = false;
                        break;
                    }
                } else if (!wait_bar(&empty[st], ((it / S) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                // segment 0: hi.hi, 1: hi.lo, 2: lo.hi
                const int seg = kbt / t.kseg;
                const int k0 = (kbt - seg * t.kseg) * kBK;
                const CUtensorMap *ma = &om.A[seg == 2 ? 1 : 0];
                const CUtensorMap *mbp = &om.B[seg == 1 ? 1 : 0];
                if (rank == 0 && lane == 0) mbar_arrive_expect_tx(&full[st], kPairTx);
                const uint32_t fb = full_even + st * 8;
                uint8_t *sa = smem + st * kStageBytes;
                uint8_t *sb = sa + kStageA;
                if (gA) {
                    tma_gather4_pair(sa + lane * 512, ma, fb, k0, rows);
                    if (lane == 0) tma_load_2d_pair(sb, mbp, fb, k0, (t.type == T_G ? a.v0n : 0) + bn);
                } else if (gB) {
                    // lanes 0-15: column block 0, lanes 16-31: block 1; 4 token rows each
                    tma_gather4_pair(sb + (lane >> 4) * kAtomBytes + (lane & 15) * 512, mbp, fb,
                                     bn + (lane >> 4) * kAtom, rows);
                    if (lane == 0) tma_load_3d_pair(sa, ma, fb, 0, k0, am / kAtom);
                } else if (lane == 0) {
                    load_operands(t, a, ma, mbp, sa, sb, fb, am, bn, k0);
                }
            }
        }
    }
    if (KIND != KIND_LSE && !dep_done) {
        // the next launch may only start once the one before this has finished
        griddep_wait();
        if (lane == 0) griddep_launch_dependents();
    }
    if (!ok && rank == 0 && lane == 0) {
        // let the copies already issued (by both CTAs) land before the pair exits
        const int first = it > S ? it - S : 0;
        for (int j = first; j < it; ++j) drain_bar(&full[j % S], (j / S) & 1);
    }
}

// One CTA pair (cluster of 2) per two SMs. Each CTA loads its 128 A rows and
// its 128 of the 256 B rows per stage; the even CTA waits for both halves on
// its full barrier, issues tcgen05.mma.cta_group::2 (M = 256, N = 256) and
// commits stage releases and accumulator-ready signals to both CTAs; each
// CTA's epilogue reads its own 128 rows from its TMEM and releases the
// accumulator with an arrive on the even CTA's barrier.
template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
    constexpr uint32_t kIdescKK = idesc_f32acc(kFmtBf16, kPairM, kBN, false, false);   // LSE, G
    constexpr uint32_t kIdescKM = idesc_f32acc(kFmtBf16, kPairM, kBN, false, true);    // DH
    constexpr uint32_t kIdescMM = idesc_f32acc(kFmtBf16, kPairM, kBN, true, true);     // DW

    constexpr int S = Cfg<KIND>::kS;          // pipeline stages
    constexpr int EW = Cfg<KIND>::kEpiWarp;   // staging bytes per epilogue warp
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *epi_stage = smem + S * kStageBytes;                                  // epilogue staging buffers
    uint64_t *full = reinterpret_cast<uint64_t *>(epi_stage + 4 * EW);             // used on the even CTA
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;                                                   // used on the even CTA
    uint64_t *mma_done = tempty + 2;
    uint64_t *opt_bar = mma_done + 1;                                               // optimizer ring (4 x 3)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(opt_bar + 4 * kOptLoadBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0 = even CTA (issues the MMAs), 1 = its peer
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int nv = a.counters[0];
    const Sched s = make_sched<KIND>(a, nv);
    if (pair >= s.units) return;   // uniform over both CTAs of the pair

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        if (KIND == KIND_BWD_OPT)
            for (int i = 0; i < 4 * kOptLoadBars; ++i) mbar_init(&opt_bar[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);   // 4 epilogue warps in each CTA of the pair
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int slot = 0; slot < (KIND == KIND_LSE ? 1 : 3); ++slot)
            for (int h = 0; h < a.nseg && h < 2; ++h) {
                tma_prefetch_map(&maps.t[slot].A[h]);
                tma_prefetch_map(&maps.t[slot].B[h]);
            }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();   // barrier inits and the TMEM allocation are visible to both CTAs
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the even CTA's full and tempty barriers, as shared::cluster addresses
    const uint32_t full_even = map_to_cta(smem_u32(full), 0);
    const uint32_t tempty_even = map_to_cta(smem_u32(tempty), 0);

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        // lane 0 alone, except with row gather, where every lane issues one
        // gather4 per stage
        if (a.gather)
            producer<KIND, true>(maps, a, s, pair, npairs, rank, lane, smem, full, empty, full_even, abort_flag);
        else if (lane == 0)
            producer<KIND, false>(maps, a, s, pair, npairs, rank, lane, smem, full, empty, full_even, abort_flag);
    } else if (warp == 1) {
        // ------------------------------------------- MMA issue (even CTA only)
        if (lane == 0 && rank == 0) {
            int it = 0, tile = 0;
            bool ok = true;
            for (int u = pair; ok && u < s.units; u += npairs) {
                int n0, n1;
                unit_range<KIND>(s, u, n0, n1);
                for (int n = n0; ok && n < n1; ++n, ++tile) {
                    const TileInfo t = tile_info<KIND>(s, u, n);
                    const bool a_mn = t.type == T_DW;
                    const bool b_mn = t.type == T_DW || t.type == T_DH;
                    const uint32_t idesc = a_mn ? kIdescMM : (b_mn ? kIdescKM : kIdescKK);
                    const int k_blocks = t.kseg * a.nseg;
                    const int acc = tile & 1;
                    if (!wait_bar(&tempty[acc], ((tile >> 1) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * kBN;
                    for (int kb = 0; kb < k_blocks; ++kb, ++it) {
                        const int st = it % S;
                        if (!wait_bar(&full[st], (it / S) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t sa = smem_u32(smem + st * kStageBytes);
                        const uint32_t sb = sa + kStageA;
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                            const uint64_t ad = a_mn ? sdesc_sw128(sa + kk * kUmmaK * 128, kAtomBytes, 1024)
                                                     : sdesc_sw128(sa + kk * 32, 16, 1024);
                            const uint64_t bd = b_mn ? sdesc_sw128(sb + kk * kUmmaK * 128, kAtomBytes, 1024)
                                                     : sdesc_sw128(sb + kk * 32, 16, 1024);
                            umma_f16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                        }
                        umma_commit_pair_mc(&empty[st], 3);   // frees the stage in both CTAs
                    }
                    if (!ok) break;
                    umma_commit_pair_mc(&tfull[acc], 3);      // accumulator ready in both CTAs
                }
            }
            umma_commit_pair_mc(mma_done, 1);
            drain_bar(mma_done, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int trow = quarter * 32 + lane;     // row within this CTA's 128 rows == TMEM lane
        uint8_t *stage_mine = epi_stage + (warp - 2) * EW;   // this warp's staging buffers
        // fused optimizer: this warp's ring of W / state boxes in its 16 KB
        // staging area: with fp32 state three 5 KB buffers, or two 8 KB ones
        // when fp32 weights move; with bf16 state five 3 KB buffers (bf16 W),
        // four of 4 KB (fp32 W) or three of 5 KB (fp32 master)
        OptRing ring{};
        if (KIND == KIND_BWD_OPT) {
            const bool w32 = a.opt.master || a.opt.w_fp32;
            ring.base = stage_mine;
            ring.bar = opt_bar + (warp - 2) * kOptLoadBars;
            // buffer bytes (1 KB multiples): the state boxes, the weights box and,
            // with a master copy, the bf16 W box it is rounded into
            ring.bsz = a.opt.s16 ? (w32 ? (a.opt.master ? 5120 : 4096) : 3072) : (w32 ? 8192 : 5120);
            ring.nbuf = EW / ring.bsz < kOptLoadBars ? EW / ring.bsz : kOptLoadBars;
            const uint32_t sb = a.opt.s16 ? 1024u : 2048u;   // one state box (16 columns x 32 rows)
            ring.bytes = ((a.opt.kind == OPT_ADAMW || a.opt.momentum != 0.f) ? sb : 0u) +
                         (a.opt.kind == OPT_ADAMW ? sb : 0u) + (w32 ? 2048u : 1024u);
        }
        int ebuf = 0;
        const float gscale = a.grad_ptr ? a.grad_scale * *a.grad_ptr : a.grad_scale;
        const int nvn = *a.nv_norm;
        const float inv_nv = nvn > 0 ? gscale / static_cast<float>(nvn) : 0.f;
        int tile = 0;
        bool ok = true;
        bool dep_done = false;
        for (int u = pair; ok && u < s.units; u += npairs) {
            int n0, n1;
            unit_range<KIND>(s, u, n0, n1);
            float run_m = -INFINITY, run_l = 0.f;   // online log-sum-exp of this row over the unit (LSE)
            int grow = 0;
            for (int n = n0; n < n1; ++n, ++tile) {
                const TileInfo t = tile_info<KIND>(s, u, n);
                if (KIND != KIND_LSE && !dep_done && t.type != T_G) {
                    griddep_wait();   // the dH accumulator / dW rows of the previous launch
                    dep_done = true;
                }
                // compacted row (LSE/G/DH) or chunk vocab row (DW) of this thread
                grow = t.mb * kPairM + static_cast<int>(rank) * kBM + trow;
                // target column relative to the first column of the vocab range
                // this tile type covers; negative / out of range when absent
                int tgt = -1;
                float lse2 = INFINITY;
                if (t.type == T_LSE) tgt = grow < nv ? a.tc[grow] : -1;
                if (t.type == T_G && grow < nv) {
                    tgt = a.tc[grow] - a.v0n;
                    lse2 = a.lse2[grow];
                }
                const int acc = tile & 1;
                const bool opt_dw = KIND == KIND_BWD_OPT && t.type == T_DW;
                // fused optimizer: this warp's 32 W rows and the tile's 16-column boxes
                // that lie inside d; the first boxes' loads do not depend on the
                // accumulator and are issued before waiting for it
                const int opt_row0 = a.v0w + t.mb * kPairM + static_cast<int>(rank) * kBM + quarter * 32;
                const int opt_col0 = t.nt * kBN;
                const int opt_np = opt_dw ? (a.d - opt_col0 >= kBN ? kBN / 16 : cdiv(a.d - opt_col0, 16)) : 0;
                if (opt_dw) {
                    if (lane == 0) {
                        bulk_wait_group_read<0>();   // earlier stores have read the staging area
                        for (int p = 0; p < ring.nbuf && p < opt_np; ++p)
                            opt_issue(maps, a.opt, ring, p, opt_col0 + 16 * p, opt_row0);
                    }
                    __syncwarp();
                }
                if (!wait_bar(&tfull[acc], (tile >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN;
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    const int col = t.nt * kBN + c * 32;   // column within the vocab range / d
                    if (opt_dw && 2 * c >= opt_np) break;   // boxes past d: nothing to update
                    uint32_t r[32];
                    tmem_ld32(tbase + c * 32, r);
                    tmem_ld_wait();
                    if (t.type == T_LSE) {
                        const int rel = tgt - col;
                        if (static_cast<unsigned>(rel) < 32u) {
                            float zv = 0.f;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (j == rel) zv = __uint_as_float(r[j]);
                            a.z[grow] = zv;
                        }
                        float x[32];
                        float cm = -INFINITY;
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            x[j] = (col + j < a.V) ? __uint_as_float(r[j]) * kLog2e : -INFINITY;
                            cm = fmaxf(cm, x[j]);
                        }
                        const float mn = fmaxf(run_m, cm);
                        if (mn != -INFINITY) {
                            float sum = 0.f;
#pragma unroll
                            for (int j = 0; j < 32; ++j) sum += exp2f(x[j] - mn);
                            run_l = run_l * exp2f(run_m - mn) + sum;
                            run_m = mn;
                        }
                    } else {
                        // G, DW, DH: values for this thread's row -> swizzled staging
                        // buffer -> one bulk tensor store (or add) of the 32x32 chunk
                        float v[32];
                        if (t.type == T_G) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                float g = exp2f(__uint_as_float(r[j]) * kLog2e - lse2) * inv_nv;
                                if (col + j == tgt) g -= inv_nv;
                                v[j] = (col + j < a.vlenn) ? g : 0.f;
                            }
                        } else {
                            const bool zero_acc = (t.kseg == 0);   // dW with no valid token
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = zero_acc ? 0.f : __uint_as_float(r[j]);
                        }
                        if (opt_dw) {
                            // fused optimizer: boxes 2c and 2c+1 (16 columns each) of the
                            // ring; lane = W row; no dW store
                            bool box_ok = true;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const int p = 2 * c + h;
                                if (p >= opt_np) break;
                                const int b = p % ring.nbuf;
                                if (!wait_bar(ring.bar + b, (ring.phase >> b) & 1u, abort_flag)) {
                                    box_ok = false;
                                    break;
                                }
                                ring.phase ^= 1u << b;
                                ring.pend &= ~(1u << b);
                                opt_row(a.opt, ring.base + b * ring.bsz, lane, v + 16 * h);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    opt_store(maps, a.opt, ring, p, opt_col0 + 16 * p, opt_row0);
                                    if (p + ring.nbuf < opt_np) {
                                        bulk_wait_group_read<0>();   // the store has read the buffer
                                        opt_issue(maps, a.opt, ring, p + ring.nbuf, opt_col0 + 16 * (p + ring.nbuf),
                                                  opt_row0);
                                    }
                                }
                                __syncwarp();
                            }
                            if (!box_ok) {
                                ok = false;
                                break;
                            }
                            continue;
                        }
                        uint8_t *sbuf = stage_mine + ebuf * kEpiBufBytes;
                        if (lane == 0) bulk_wait_group_read<1>();   // this buffer's store of two chunks ago has read it
                        __syncwarp();
                        if (t.type == T_G || (t.type == T_DW && a.dw_bf16)) {
                            // bf16 rows of 64 bytes; 16-byte unit k of row `lane` at unit k ^ ((lane >> 1) & 3)
                            float lo[32];
                            if (a.nseg > 1) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) split_bf16(v[j], v[j], lo[j]);
                            }
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int off = lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4);
                                *reinterpret_cast<uint4 *>(sbuf + off) =
                                    make_uint4(pack_bf16x2(v[8 * k], v[8 * k + 1]), pack_bf16x2(v[8 * k + 2], v[8 * k + 3]),
                                               pack_bf16x2(v[8 * k + 4], v[8 * k + 5]),
                                               pack_bf16x2(v[8 * k + 6], v[8 * k + 7]));
                                if (a.nseg > 1)
                                    *reinterpret_cast<uint4 *>(sbuf + 2048 + off) = make_uint4(
                                        pack_bf16x2(lo[8 * k], lo[8 * k + 1]), pack_bf16x2(lo[8 * k + 2], lo[8 * k + 3]),
                                        pack_bf16x2(lo[8 * k + 4], lo[8 * k + 5]), pack_bf16x2(lo[8 * k + 6], lo[8 * k + 7]));
                            }
                        } else {
                            // fp32 rows of 128 bytes; 16-byte unit k of row `lane` at unit k ^ (lane & 7)
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                *reinterpret_cast<float4 *>(sbuf + lane * 128 + ((k ^ (lane & 7)) << 4)) =
                                    make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int row0 = t.mb * kPairM + static_cast<int>(rank) * kBM + quarter * 32;
                            if (t.type == T_G) {
                                tma_store_2d(&maps.st_g[0], sbuf, col, row0);
                                if (a.nseg > 1) tma_store_2d(&maps.st_g[1], sbuf + 2048, col, row0);
                            } else if (t.type == T_DW) {
                                // rows past V (last chunk) are clipped by the map
                                if (a.acc_dw)
                                    tma_reduce_add_2d(&maps.st_dw, sbuf, col, a.v0w + row0);
                                else
                                    tma_store_2d(&maps.st_dw, sbuf, col, a.v0w + row0);
                            } else {
                                if (a.acc_dh)
                                    tma_reduce_add_2d(&maps.st_dh, sbuf, col, row0);
                                else
                                    tma_store_2d(&maps.st_dh, sbuf, col, row0);
                            }
                            bulk_commit_group();
                        }
                        ebuf ^= 1;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_even + acc * 8);
                if (opt_dw) {
                    // the ring overlaps the staging buffers the next tiles write
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                }
            }
            if (KIND == KIND_LSE && ok && grow < nv) {
                int split, mbu;
                lse_unit(s.m_blocks, s.splits, s.rgroup, u, split, mbu);
                a.part[static_cast<size_t>(split) * s.m_blocks * kPairM + grow] = make_float2(run_m, run_l);
            }
        }
        if (KIND == KIND_BWD_OPT && lane == 0) {
            // after an abort: let optimizer loads still in flight land first
            for (int b = 0; b < ring.nbuf; ++b)
                if (ring.pend & (1u << b)) drain_bar(ring.bar + b, (ring.phase >> b) & 1u);
        }
        if (lane == 0) bulk_wait_group_all();   // this warp's stores have written global memory
    }

    // Both CTAs stay resident until every remote arrive, multicast commit and
    // copy aimed at either of them has landed; then the pair frees its TMEM.
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

}  // namespace lce
