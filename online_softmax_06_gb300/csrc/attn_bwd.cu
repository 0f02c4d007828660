// attn_bwd.cu -- attention backward (dQ, dK, dV) on the sm_103a tensor cores.
//
// What it computes: the gradients of sum(dO * O) for O = softmax(scale Q K^T +
// mask) V, with the probabilities recomputed tile by tile from the forward's
// row logsumexp instead of being stored ("少搬一趟：FlashAttention 四代进化史"
// §2.4: P_ij = exp(S_ij - L_i); "第二十二课：Softmax 为什么难以高效…" §三十-三十一):
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),   D_i = dO_i . O_i,
//     dQ = scale dS K,   dK = scale dS^T Q.
// The booklet's §3.3 splits the backward over K/V column blocks and sums the
// overlapping dQ contributions with atomic adds; here a K/V block's CTA needs
// all 512 tensor-memory columns for S^T, dP^T, dV and dK (d = 128), so dQ has
// its own pass over Q row blocks instead (no atomics, deterministic), at the
// cost of recomputing S and dP there.
//
// Two kernels, launched in this order on one stream:
//   * attn_bwd_dq_kernel: one CTA per (sequence, head, 128-query tile).  Each
//     query row is served by two threads (64 columns each): they form
//     D_i = dO_i . O_i (stored for the second kernel), then for every visible key tile j
//     turns S = Q K_j^T and dP = dO V_j^T (tcgen05, fp32 in TMEM) into
//     dS = P o (dP - D_i) in bf16 in TMEM, and the MMA warp accumulates
//     dQ += dS K_j in TMEM.
//   * attn_bwd_dkdv_kernel: one CTA per (sequence, head, 128-key tile), K and
//     V resident in shared memory.  For every query tile i that sees the keys,
//     S^T = K Q_i^T and dP^T = V dO_i^T land in TMEM with one key per TMEM
//     lane; the two threads of each key row form P^T and dS^T
//     (bf16, in TMEM) from the query tile's logsumexp and D (staged in shared
//     memory by the load warp), and the MMA warp accumulates dV += P^T dO_i and
//     dK += dS^T Q_i.
// The elementwise work (P, dS) needs no reduction along a row, so a row's 128
// columns are split between two threads: warps 0-7 serve the rows (warp w:
// TMEM lanes 32 (w % 4) .. + 31, columns 64 (w / 4) .. + 63), which hides
// more of the exp and TMEM latencies than one thread per row.  Warp 8 issues
// TMA loads into a ring of shared-memory stages and warp 9 owns the tensor
// memory and issues every tcgen05.mma.  Every wait is
// bounded; a wait that gives up raises the error word and the abort flag, the
// roles leave their loops, in-flight copies and MMAs drain, and the CTA frees
// its tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_error.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BT = 128;                     // rows of a Q, K, V or dO tile
constexpr int G = 2;                        // threads per row (column groups)
constexpr int kColsPerThread = BT / G;
constexpr int kRowWarps = 4 * G;
constexpr int kThreads = 32 * (kRowWarps + 2);
constexpr int kWarpLoad = kRowWarps;
constexpr int kWarpMma = kRowWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kChunkBytes = BT * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = BT * D * 2;
    static constexpr int kStages = 4;        // two per step (even / odd positions)
    // shared memory: [A0][A1][ring x kStages][stats: 2 slots x (lse2, D) x 128
    // floats][barriers, flags]
    static constexpr uint32_t kOffA0 = 0;
    static constexpr uint32_t kOffA1 = kTileBytes;
    static constexpr uint32_t kOffRing = 2 * kTileBytes;
    static constexpr uint32_t kOffStat = kOffRing + kStages * kTileBytes;
    static constexpr uint32_t kStatBytes = 2 * 2 * BT * 4;
    static constexpr uint32_t kOffBar = kOffStat + kStatBytes;
    // a_full, kv_full[S], kv_empty[S], s_full, p_full, o_full, drain
    static constexpr uint32_t kBarBytes = 8 * (1 + 2 * kStages + 4);
    static constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 16 + 1024;
};

// TMEM columns: S (or S^T) [0, 128), dP (or dP^T) [128, 256), accumulators from
// 256 (dQ; or dV then dK).  bf16 P / dS are packed into the region they are
// formed from: the 32 values of each 32-column block go to the block's first 16
// columns (two per column), so a thread only overwrites columns it has read.
constexpr uint32_t kColS = 0, kColP = 128, kColAcc = 256;
// Column of the packed bf16 operand for the MMA's K step kk (16 values).
__host__ __device__ constexpr uint32_t packed_col(int kk)
{
    return uint32_t(32 * (kk >> 1) + 8 * (kk & 1));
}

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;    // [B*N, H, d] bf16, box {64, 1, 128}
    const __nv_bfloat16 *O, *dO;
    const float *lse;                       // [B, H, N], natural log
    float *D;                               // [B, H, N]
    __nv_bfloat16 *dQ, *dK, *dV;
    int B, H, N, n_tiles;
    float scale, scale_log2;
    int causal;
    int *err_word;
};

struct Bars {
    uint64_t *a_full, *kv_full, *kv_empty, *s_full, *p_full, *o_full, *drain;
};

template <int D>
__device__ __forceinline__ Bars carve(uint8_t *smem)
{
    using C = Cfg<D>;
    uint64_t *b = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    Bars r;
    r.a_full = b;
    r.kv_full = b + 1;
    r.kv_empty = b + 1 + C::kStages;
    r.s_full = b + 1 + 2 * C::kStages;
    r.p_full = r.s_full + 1;
    r.o_full = r.s_full + 2;
    r.drain = r.s_full + 3;
    return r;
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 0; it < kWaitMaxPolls; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return;
        if ((it & 255u) == 255u && ptx::globaltimer() - t0 > kWaitTimeoutNs)
            return;
    }
}

// Shared set-up of both kernels: barriers, tensor memory, tensor-map prefetch.
// kv_full of odd ring positions counts `odd_arrivals` arrivals (the load warp's
// lanes stage statistics with those tiles in the dK/dV kernel).
template <int D>
__device__ __forceinline__ uint32_t setup(const BwdParams &p, uint8_t *smem, const Bars &bar,
                                          uint32_t odd_arrivals, volatile int *abort_flag,
                                          uint32_t *tmem_slot)
{
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar.a_full, 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bar.kv_full[s], (s & 1) ? odd_arrivals : 1u);
            ptx::mbar_init(&bar.kv_empty[s], 1);
        }
        ptx::mbar_init(bar.s_full, 1);
        ptx::mbar_init(bar.p_full, BT * G);
        ptx::mbar_init(bar.o_full, 1);
        ptx::mbar_init(bar.drain, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        ptx::prefetch_tmap(&p.tm_q);
        ptx::prefetch_tmap(&p.tm_k);
        ptx::prefetch_tmap(&p.tm_v);
        ptx::prefetch_tmap(&p.tm_do);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    (void)smem;
    return *tmem_slot;
}

template <int D>
__device__ __forceinline__ void teardown(uint32_t tmem)
{
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if ((threadIdx.x >> 5) == kWarpMma)
        ptx::tmem_dealloc(tmem, kTmemCols);
}

// Row `r` of a 128-row tile's accumulator (32-bit TMEM columns [col, col + D))
// scaled by `mul`, written as bf16 to dst (one row of D elements).
template <int D>
__device__ __forceinline__ void store_row(uint32_t t_acc, float mul, __nv_bfloat16 *dst, bool ok)
{
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(t_acc + c * 32, o);
        ptx::tmem_wait_ld();
        if (ok) {
            uint4 *out = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 0]) * mul,
                                       __uint_as_float(o[8 * q + 1]) * mul);
                w.y = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2]) * mul,
                                       __uint_as_float(o[8 * q + 3]) * mul);
                w.z = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 4]) * mul,
                                       __uint_as_float(o[8 * q + 5]) * mul);
                w.w = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 6]) * mul,
                                       __uint_as_float(o[8 * q + 7]) * mul);
                out[q] = w;
            }
        }
    }
}

// =============================================================================
// dQ (and D) -- one CTA per (sequence, head, query tile), heaviest tiles first
// =============================================================================
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Bars bar = carve<D>(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + C::kBarBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int bh_count = p.B * p.H;
    const int qt = p.n_tiles - 1 - int(blockIdx.x) / bh_count;
    const int bh = int(blockIdx.x) % bh_count;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t row0 = int64_t(b) * p.N;          // first row of the sequence
    const int n_kv = p.causal ? qt + 1 : p.n_tiles;  // key tiles this query tile sees
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t tmem = setup<D>(p, smem, bar, 1u, abort_flag, tmem_slot);
    bool aborted = false;
    uint8_t *tile_q = smem + C::kOffA0, *tile_do = smem + C::kOffA1;
    uint8_t *ring = smem + C::kOffRing;

    if (warp == kWarpLoad) {
        // ======================= TMA producer ==============================
        if (lane == 0) {
            int last_phase[C::kStages];
            for (int s = 0; s < C::kStages; ++s)
                last_phase[s] = -1;
            ptx::mbar_arrive_expect_tx(bar.a_full, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                ptx::tma_load_3d(tile_q + c * kChunkBytes, &p.tm_q, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(qt) * BT));
                ptx::tma_load_3d(tile_do + c * kChunkBytes, &p.tm_do, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(qt) * BT));
            }
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < n_kv && !aborted; ++j) {
                for (int kv = 0; kv < 2; ++kv) {
                    if (!ptx::mbar_wait(&bar.kv_empty[stage], phase ^ 1u, abort_flag,
                                        p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&bar.kv_full[stage], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(ring + stage * C::kTileBytes + c * kChunkBytes,
                                         kv ? &p.tm_v : &p.tm_k, &bar.kv_full[stage], c * 64, h,
                                         int(row0 + int64_t(j) * BT));
                    last_phase[stage] = int(phase);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (aborted || *abort_flag) {
                drain_wait(bar.a_full, 0);
                for (int s = 0; s < C::kStages; ++s)
                    if (last_phase[s] >= 0)
                        drain_wait(&bar.kv_full[s], uint32_t(last_phase[s]));
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer ================================
        if (lane == 0) {
            constexpr uint32_t idesc_ss = ptx::idesc_bf16_f32(BT, BT, false);
            constexpr uint32_t idesc_ts = ptx::idesc_bf16_f32(BT, D, true);
            constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
            constexpr uint64_t desc_mnmajor = ptx::smem_desc_base(kChunkBytes, 1024);
            const uint64_t dq = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_q));
            const uint64_t ddo = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_do));
            const uint32_t ring_addr = ptx::smem_u32(ring);
            int stage = 0;
            uint32_t phase = 0;
            auto advance = [&]() {
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            do {
                if (!ptx::mbar_wait(bar.a_full, 0, abort_flag, p.err_word)) {
                    aborted = true;
                    break;
                }
                for (int j = 0; j < n_kv; ++j) {
                    // S = Q K_j^T
                    if (!ptx::mbar_wait(&bar.kv_full[stage], phase, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    const int k_stage = stage;
                    const uint32_t k_addr = ring_addr + stage * C::kTileBytes;
                    advance();
                    ptx::tc_fence_after_sync();
                    const uint64_t dk = ptx::smem_desc(desc_kmajor, k_addr);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(tmem + kColS, dq + off, dk + off, idesc_ss, kk > 0 ? 1u : 0u);
                    }
                    // dP = dO V_j^T
                    if (!ptx::mbar_wait(&bar.kv_full[stage], phase, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    const int v_stage = stage;
                    const uint64_t dv =
                        ptx::smem_desc(desc_kmajor, ring_addr + stage * C::kTileBytes);
                    advance();
                    ptx::tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(tmem + kColP, ddo + off, dv + off, idesc_ss, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar.s_full);
                    ptx::mma_commit(&bar.kv_empty[v_stage]);
                    // dQ += dS K_j   (dS: bf16 over the first 64 columns of S)
                    if (!ptx::mbar_wait(bar.p_full, uint32_t(j) & 1u, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t dkn = ptx::smem_desc(desc_mnmajor, k_addr);
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc, tmem + kColS + packed_col(kk),
                                    dkn + uint64_t((kk * 16 * 128) >> 4), idesc_ts,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(&bar.kv_empty[k_stage]);
                }
                if (!aborted)
                    ptx::mma_commit(bar.o_full);
            } while (false);
            ptx::mma_commit(bar.drain);
            drain_wait(bar.drain, 0);
        }
        __syncwarp();
    } else {
        // ======================= query rows ================================
        const int r = (warp & 3) * 32 + lane;        // query row in the tile = TMEM lane
        const int g = warp >> 2;                     // column group
        const int i = qt * BT + r;
        const bool row_ok = i < p.N;
        const uint32_t lane_bits = uint32_t((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_bits + kColS;
        const uint32_t tP = tmem + lane_bits + kColP;
        const int64_t stat = (int64_t(b) * p.H + h) * p.N + i;
        // D_i = dO_i . O_i (fp32); group 0 stores it for the dK/dV kernel
        float Di = 0.f, lse2 = 0.f;
        if (row_ok) {
            const uint4 *o4 = reinterpret_cast<const uint4 *>(p.O + ((row0 + i) * p.H + h) * D);
            const uint4 *g4 = reinterpret_cast<const uint4 *>(p.dO + ((row0 + i) * p.H + h) * D);
#pragma unroll 4
            for (int u = 0; u < D / 8; ++u) {
                const uint4 ov = o4[u], gv = g4[u];
                const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 of =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[e]));
                    const float2 gf =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[e]));
                    Di = fmaf(of.x, gf.x, Di);
                    Di = fmaf(of.y, gf.y, Di);
                }
            }
            if (g == 0)
                p.D[stat] = Di;
            lse2 = p.lse[stat] * kLog2e;
        }
        const float sl = p.scale_log2;

        for (int j = 0; j < n_kv; ++j) {
            if (!ptx::mbar_wait(bar.s_full, uint32_t(j) & 1u, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            // last visible column of this key tile for row i (causal diagonal,
            // end of the sequence); rows past the end see nothing
            const bool diag = p.causal && j == qt;
            int lim = diag ? r : BT - 1;
            const int lim_len = p.N - 1 - j * BT;
            if (lim_len < lim)
                lim = lim_len;
            if (!row_ok)
                lim = -1;
#pragma unroll
            for (int blk = 0; blk < kColsPerThread / 32; ++blk) {
                const int col0 = g * kColsPerThread + blk * 32;
                uint32_t sv[32], dv[32], pk[16];
                ptx::tmem_ld32(tS + col0, sv);
                ptx::tmem_ld32(tP + col0, dv);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float ds[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int c = col0 + 2 * e + k;
                        const float x = __uint_as_float(sv[2 * e + k]);
                        const float y = __uint_as_float(dv[2 * e + k]);
                        // masked entries get exponent -inf: exp2 gives 0, no branch
                        const float pv = ptx::ex2(c <= lim ? fmaf(x, sl, -lse2) : -INFINITY);
                        ds[k] = pv * (y - Di);
                    }
                    pk[e] = ptx::pack_bf16x2(ds[0], ds[1]);
                }
                ptx::tmem_st16(tS + col0, pk);        // dS of this block, packed
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar.p_full);
        }
        // the epilogue reads each row's dQ once: group 0 stores it
        if (!aborted && ptx::mbar_wait(bar.o_full, 0, abort_flag, p.err_word)) {
            ptx::tc_fence_after_sync();
            if (g == 0)
                store_row<D>(tmem + lane_bits + kColAcc, p.scale,
                             p.dQ + ((row0 + i) * p.H + h) * D, row_ok);
        }
    }
    teardown<D>(tmem);
}

// =============================================================================
// dK, dV -- one CTA per (sequence, head, key tile), heaviest tiles first
// =============================================================================
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p)
{
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Bars bar = carve<D>(smem);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + C::kBarBytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int bh_count = p.B * p.H;
    const int kt = int(blockIdx.x) / bh_count;       // causal: low key tiles see most
    const int bh = int(blockIdx.x) % bh_count;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t row0 = int64_t(b) * p.N;
    const int i0 = p.causal ? kt : 0;                // first query tile that sees the keys
    const int n_q = p.n_tiles - i0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t tmem = setup<D>(p, smem, bar, 32u, abort_flag, tmem_slot);
    bool aborted = false;
    uint8_t *tile_k = smem + C::kOffA0, *tile_v = smem + C::kOffA1;
    uint8_t *ring = smem + C::kOffRing;
    float *stats = reinterpret_cast<float *>(smem + C::kOffStat);   // slot x (lse2, D) x 128

    if (warp == kWarpLoad) {
        // ======================= TMA producer (whole warp) ===================
        // Ring positions 2s and 2s + 1 hold Q_i and dO_i of step s (i = i0 + s);
        // with dO_i the warp's lanes also stage the tile's log2 logsumexp and D.
        int last_phase[C::kStages];
        for (int s = 0; s < C::kStages; ++s)
            last_phase[s] = -1;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar.a_full, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                ptx::tma_load_3d(tile_k + c * kChunkBytes, &p.tm_k, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
                ptx::tma_load_3d(tile_v + c * kChunkBytes, &p.tm_v, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
            }
        }
        int stage = 0;
        uint32_t phase = 0;
        const int64_t stat0 = (int64_t(b) * p.H + h) * p.N;
        for (int s = 0; s < n_q && !aborted; ++s) {
            const int i = i0 + s;
            for (int kv = 0; kv < 2; ++kv) {
                int ok = 1;
                if (lane == 0)
                    ok = ptx::mbar_wait(&bar.kv_empty[stage], phase ^ 1u, abort_flag, p.err_word)
                             ? 1
                             : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    aborted = true;
                    break;
                }
                if (kv == 1) {
                    float *slot = stats + (stage >> 1) * (2 * BT);
#pragma unroll
                    for (int u = 0; u < BT / 32; ++u) {
                        const int c = lane * (BT / 32) + u;
                        const int q = i * BT + c;
                        const bool v = q < p.N;
                        slot[c] = v ? p.lse[stat0 + q] * kLog2e : 0.f;
                        slot[BT + c] = v ? p.D[stat0 + q] : 0.f;
                    }
                }
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&bar.kv_full[stage], C::kTileBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        ptx::tma_load_3d(ring + stage * C::kTileBytes + c * kChunkBytes,
                                         kv ? &p.tm_do : &p.tm_q, &bar.kv_full[stage], c * 64, h,
                                         int(row0 + int64_t(i) * BT));
                    last_phase[stage] = int(phase);
                } else if (kv == 1) {
                    ptx::mbar_arrive(&bar.kv_full[stage]);
                }
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (lane == 0 && (aborted || *abort_flag)) {
            drain_wait(bar.a_full, 0);
            for (int s = 0; s < C::kStages; ++s)
                if (last_phase[s] >= 0)
                    drain_wait(&bar.kv_full[s], uint32_t(last_phase[s]));
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer ================================
        if (lane == 0) {
            constexpr uint32_t idesc_ss = ptx::idesc_bf16_f32(BT, BT, false);
            constexpr uint32_t idesc_ts = ptx::idesc_bf16_f32(BT, D, true);
            constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
            constexpr uint64_t desc_mnmajor = ptx::smem_desc_base(kChunkBytes, 1024);
            const uint64_t dk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_k));
            const uint64_t dvk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_v));
            const uint32_t ring_addr = ptx::smem_u32(ring);
            int stage = 0;
            uint32_t phase = 0;
            auto advance = [&]() {
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            do {
                if (!ptx::mbar_wait(bar.a_full, 0, abort_flag, p.err_word)) {
                    aborted = true;
                    break;
                }
                for (int s = 0; s < n_q; ++s) {
                    // S^T = K Q_i^T
                    if (!ptx::mbar_wait(&bar.kv_full[stage], phase, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    const int q_stage = stage;
                    const uint32_t q_addr = ring_addr + stage * C::kTileBytes;
                    advance();
                    ptx::tc_fence_after_sync();
                    const uint64_t dq = ptx::smem_desc(desc_kmajor, q_addr);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(tmem + kColS, dk + off, dq + off, idesc_ss, kk > 0 ? 1u : 0u);
                    }
                    // dP^T = V dO_i^T
                    if (!ptx::mbar_wait(&bar.kv_full[stage], phase, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    const int do_stage = stage;
                    const uint32_t do_addr = ring_addr + stage * C::kTileBytes;
                    advance();
                    ptx::tc_fence_after_sync();
                    const uint64_t ddo = ptx::smem_desc(desc_kmajor, do_addr);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(tmem + kColP, dvk + off, ddo + off, idesc_ss, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(bar.s_full);
                    // dV += P^T dO_i,  dK += dS^T Q_i
                    if (!ptx::mbar_wait(bar.p_full, uint32_t(s) & 1u, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint64_t ddo_mn = ptx::smem_desc(desc_mnmajor, do_addr);
                    const uint64_t dq_mn = ptx::smem_desc(desc_mnmajor, q_addr);
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc, tmem + kColS + packed_col(kk),
                                    ddo_mn + uint64_t((kk * 16 * 128) >> 4), idesc_ts,
                                    (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc + D, tmem + kColP + packed_col(kk),
                                    dq_mn + uint64_t((kk * 16 * 128) >> 4), idesc_ts,
                                    (s > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(&bar.kv_empty[q_stage]);
                    ptx::mma_commit(&bar.kv_empty[do_stage]);
                }
                if (!aborted)
                    ptx::mma_commit(bar.o_full);
            } while (false);
            ptx::mma_commit(bar.drain);
            drain_wait(bar.drain, 0);
        }
        __syncwarp();
    } else {
        // ======================= key rows ==================================
        const int r = (warp & 3) * 32 + lane;        // key row in the tile = TMEM lane
        const int g = warp >> 2;                     // column group
        const int k = kt * BT + r;
        const uint32_t lane_bits = uint32_t((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_bits + kColS;
        const uint32_t tP = tmem + lane_bits + kColP;
        const float sl = p.scale_log2;
        for (int s = 0; s < n_q; ++s) {
            const int i = i0 + s;
            // the statistics arrive with dO_i at ring position 2s + 1
            const int pos = 2 * s + 1;
            const int st = pos % C::kStages;
            if (!ptx::mbar_wait(bar.s_full, uint32_t(s) & 1u, abort_flag, p.err_word) ||
                !ptx::mbar_wait(&bar.kv_full[st], uint32_t(pos / C::kStages) & 1u, abort_flag,
                                p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            const float *lse2s = stats + (st >> 1) * (2 * BT);
            const float *Ds = lse2s + BT;
            // visible columns [lo, hi]: causal keeps queries >= the key; the
            // sequence ends at N
            const int lo = (p.causal && i == kt) ? r : 0;
            int hi = p.N - 1 - i * BT;
            if (hi > BT - 1)
                hi = BT - 1;
#pragma unroll
            for (int blk = 0; blk < kColsPerThread / 32; ++blk) {
                const int col0 = g * kColsPerThread + blk * 32;
                uint32_t sv[32], dv[32], pk[16], dk[16];
                ptx::tmem_ld32(tS + col0, sv);
                ptx::tmem_ld32(tP + col0, dv);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const int c0 = col0 + 4 * e4;
                    const float4 l4 = *reinterpret_cast<const float4 *>(lse2s + c0);
                    const float4 d4 = *reinterpret_cast<const float4 *>(Ds + c0);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                    const float dd[4] = {d4.x, d4.y, d4.z, d4.w};
                    float pv[4], ds[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c = c0 + u;
                        const float x = __uint_as_float(sv[4 * e4 + u]);
                        const float y = __uint_as_float(dv[4 * e4 + u]);
                        // masked entries get exponent -inf: exp2 gives 0, no branch
                        pv[u] = ptx::ex2((c >= lo && c <= hi) ? fmaf(x, sl, -lv[u]) : -INFINITY);
                        ds[u] = pv[u] * (y - dd[u]);
                    }
                    pk[2 * e4] = ptx::pack_bf16x2(pv[0], pv[1]);
                    pk[2 * e4 + 1] = ptx::pack_bf16x2(pv[2], pv[3]);
                    dk[2 * e4] = ptx::pack_bf16x2(ds[0], ds[1]);
                    dk[2 * e4 + 1] = ptx::pack_bf16x2(ds[2], ds[3]);
                }
                ptx::tmem_st16(tS + col0, pk);        // P^T of this block, packed
                ptx::tmem_st16(tP + col0, dk);        // dS^T of this block, packed
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(bar.p_full);
        }
        if (!aborted && ptx::mbar_wait(bar.o_full, 0, abort_flag, p.err_word)) {
            ptx::tc_fence_after_sync();
            const bool key_ok = k < p.N;
            // group 0 writes dV, group 1 writes dK
            if (g == 0)
                store_row<D>(tmem + lane_bits + kColAcc, 1.f, p.dV + ((row0 + k) * p.H + h) * D,
                             key_ok);
            if (g == 1)
                store_row<D>(tmem + lane_bits + kColAcc + D, p.scale,
                             p.dK + ((row0 + k) * p.H + h) * D, key_ok);
        }
    }
    teardown<D>(tmem);
}

template <int D>
int launch_bwd_d(const BwdParams &p, cudaStream_t stream)
{
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(Cfg<D>::kSmemBytes));
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            int(Cfg<D>::kSmemBytes));
    });
    if (attr_err != cudaSuccess)
        return FA_ERR_CUDA;
    const int64_t blocks = int64_t(p.n_tiles) * p.B * p.H;
    attn_bwd_dq_kernel<D><<<dim3(unsigned(blocks)), dim3(kThreads), Cfg<D>::kSmemBytes, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    attn_bwd_dkdv_kernel<D>
        <<<dim3(unsigned(blocks)), dim3(kThreads), Cfg<D>::kSmemBytes, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int launch_attention_bwd(const AttnBwdArgs &a, cudaStream_t stream)
{
    BwdParams p;
    const int64_t total = int64_t(a.B) * a.N;
    if (!make_tmap_bf16(&p.tm_q, a.Q, total, a.H, a.d) ||
        !make_tmap_bf16(&p.tm_k, a.K, total, a.H, a.d) ||
        !make_tmap_bf16(&p.tm_v, a.V, total, a.H, a.d) ||
        !make_tmap_bf16(&p.tm_do, a.dO, total, a.H, a.d))
        return FA_ERR_CUDA;
    p.O = static_cast<const __nv_bfloat16 *>(a.O);
    p.dO = static_cast<const __nv_bfloat16 *>(a.dO);
    p.lse = a.lse;
    p.D = a.D;
    p.dQ = static_cast<__nv_bfloat16 *>(a.dQ);
    p.dK = static_cast<__nv_bfloat16 *>(a.dK);
    p.dV = static_cast<__nv_bfloat16 *>(a.dV);
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.n_tiles = (a.N + BT - 1) / BT;
    p.scale = a.scale;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.err_word = a.err_word;
    const int64_t blocks = int64_t(p.n_tiles) * a.B * a.H;
    if (blocks == 0)
        return FA_OK;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    return a.d == 64 ? launch_bwd_d<64>(p, stream) : launch_bwd_d<128>(p, stream);
}

}  // namespace fa
