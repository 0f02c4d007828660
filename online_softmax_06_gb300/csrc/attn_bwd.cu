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
// Two kernels, launched in this order on one stream; each keeps one 128-row
// tile resident and streams the other operand:
//   * attn_bwd_dq_kernel: one CTA per (sequence, head, 128-query tile).  The
//     row warps first copy Q and dO from their resident shared-memory tiles
//     into TMEM (the A operands of S = Q K_j^T and dP = dO V_j^T) and form
//     D_i = dO_i . O_i together (O rows from global memory; stored for the
//     second kernel).  Keys stream in 128-row steps through a 3-stage ring
//     (the third stage reuses the Q / dO region once the prologue is done);
//     S and dP are single-buffered in TMEM and the MMA warp issues S_{j+1} as
//     soon as the rows have read S_j, dQ += dS_j K_j once they have stored
//     dS_j (bf16, in TMEM), then dP_{j+1}.  Each query row is served by two
//     threads (64 columns of a step each).
//   * attn_bwd_dkdv_kernel: one CTA per (sequence, head, 128-key tile), K and
//     V resident, queries streamed in 64-row sub-tiles.  For every sub-tile i
//     that sees the keys, S^T = K Q_i^T and dP^T = V dO_i^T land in TMEM with
//     one key per TMEM lane; the two threads of each key row form P^T and
//     dS^T (bf16, in TMEM) from the sub-tile's logsumexp and D (staged in
//     shared memory by the load warp), and the MMA warp accumulates
//     dV += P^T dO_i and dK += dS^T Q_i.  S^T and dP^T of a step live in one
//     of two TMEM buffers (columns [0, 128) and [128, 256)), so the MMA warp
//     computes step s + 1's while the row threads turn step s's into P^T and
//     dS^T; the accumulators take columns [256, 512).  A sub-tile row's 64
//     columns are split between two threads: warp w serves TMEM lanes
//     32 (w % 4) .. + 31, columns 32 (w / 4) .. + 31 of the buffer.
// Warps 0-7 serve the rows; warp 8 issues TMA loads (one ring stage per step,
// each step prefetched into L2 a few steps before its load); warp 9 owns the
// tensor memory and issues every tcgen05.mma: the whole warp runs the issuing
// loop converged and one elected lane issues.
// Every wait is bounded; a wait that gives up raises the error word and the
// abort flag, the roles leave their loops, in-flight copies and MMAs drain,
// and the CTA frees its tensor memory.
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

constexpr int BT = 128;                     // rows of the resident tile
constexpr int BS = 64;                      // rows of a streamed sub-tile
constexpr int G = 2;                        // threads per row (column groups)
constexpr int kColsPerThread = BS / G;      // one 32-column block per step
constexpr int kRowWarps = 4 * G;
constexpr int kThreads = 32 * (kRowWarps + 2);
constexpr int kWarpLoad = kRowWarps;
constexpr int kWarpMma = kRowWarps + 1;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kResChunkBytes = BT * 128;  // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kSubChunkBytes = BS * 128;  // 64 rows x 128 bytes
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kL2Ahead = 4;                 // streamed sub-tiles are prefetched into L2
                                            // this many steps before their load

template <int D>
struct Cfg {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kResBytes = BT * D * 2;
    static constexpr uint32_t kSubBytes = BS * D * 2;
    // a ring stage holds one step's pair of sub-tiles, (K_j, V_j) or
    // (Q_i, dO_i), behind one barrier
    static constexpr int kStages = 4;
    static constexpr uint32_t kStageBytes = 2 * kSubBytes;
    // shared memory: [A0][A1][ring x kStages][stats: kStages slots x
    // (lse2, D) x 64 floats][barriers, flags]
    static constexpr uint32_t kOffA0 = 0;
    static constexpr uint32_t kOffA1 = kResBytes;
    static constexpr uint32_t kOffRing = 2 * kResBytes;
    static constexpr uint32_t kOffStat = kOffRing + kStages * kStageBytes;
    static constexpr uint32_t kStatBytes = kStages * 2 * BS * 4;
    static constexpr uint32_t kOffBar = kOffStat + kStatBytes;
    // a_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full, drain, a_tm
    static constexpr uint32_t kBarBytes = 8 * (1 + 2 * kStages + 7);
    static constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// TMEM columns: buffer b holds S (or S^T) in [128 b, 128 b + 64) and dP (or
// dP^T) in [128 b + 64, 128 b + 128); accumulators from 256 (dQ, then Q and
// dO as bf16 A operands; or dV then dK).  bf16 P / dS are packed into the region they are formed from: the 32
// values of each 32-column block go to the block's first 16 columns (two per
// column), so a thread only overwrites columns it has read.
constexpr uint32_t kColBuf = 128, kColDP = 64, kColAcc = 256;
// Column of the packed bf16 operand for the MMA's K step kk (16 values).
__host__ __device__ constexpr uint32_t packed_col(int kk)
{
    return uint32_t(32 * (kk >> 1) + 8 * (kk & 1));
}

// The dQ kernel's resident pair is (Q, dO) and its streamed pair (K, V); the
// dK/dV kernel's resident pair is (K, V) and its streamed pair (Q, dO).
struct BwdParams {
    CUtensorMap tm_a0, tm_a1;               // resident, [B*N, H, d] bf16, box {64, 1, 128}
    CUtensorMap tm_s0, tm_s1;               // streamed, box {64, 1, 64}
    const __nv_bfloat16 *O, *dO;
    const float *lse;                       // [B, H, N], natural log
    float *D;                               // [B, H, N]
    __nv_bfloat16 *dQ, *dK, *dV;
    int B, H, N, n_tiles, n_sub;     // N: sequence length (dense) / longest sequence (packed)
    float scale, scale_log2;
    int causal;
    int *err_word;
    const int32_t *cu_seqlens;       // packed batches: [B + 1] prefix sums (else nullptr)
    int64_t total;                   // rows of the tensors
    float *dq_acc;                   // one-pass kernel: fp32 [B * H, n_pad, d] (packed:
                                     // [H, total_pad, d])
    const float2 *stat2;             // one-pass kernel: (lse log2 e, D) pairs [B * H, n_pad]
                                     // (packed: [H, B, n_pad])
    int64_t n_pad;                   // N rounded up to 64
    int64_t total_pad;               // packed: total + 64 (a last sub-tile's reach)
    int head_groups;                 // one-pass kernel: the (sequence, head) pairs in this
                                     // many consecutive groups, heaviest key tiles first
    uint32_t expire_wait_ns;         // one-pass kernel, failure-detection test only (0: off)
};

// Rows of sequence b: its first row, its length and the index of its first
// row statistic (lse, D) for head h -- [B, H, N] dense, [H, total] packed.
// A packed length that contradicts N or the tensors is flagged, not computed.
struct SeqRows {
    int64_t row0, stat0;
    int L;
};
template <bool PACKED>
__device__ __forceinline__ bool seq_rows(const BwdParams &p, int b, int h, SeqRows &q)
{
    if constexpr (!PACKED) {
        q.row0 = int64_t(b) * p.N;
        q.L = p.N;
        q.stat0 = (int64_t(b) * p.H + h) * p.N;
        return true;
    }
    const int64_t s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
    if (s0 < 0 || s1 < s0 || s1 > p.total || s1 - s0 > p.N) {
        if (threadIdx.x == 0)
            record_device_error(p.err_word, FA_DEVERR_BAD_SEQLENS);
        return false;
    }
    q.row0 = s0;
    q.L = int(s1 - s0);
    q.stat0 = int64_t(h) * p.total + s0;
    return true;
}

struct Bars {
    uint64_t *a_full, *kv_full, *kv_empty, *s_full, *p_full, *o_full, *drain;
    uint64_t *a_tm;                          // dQ kernel: Q and dO copied into TMEM
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
    r.s_full = b + 1 + 2 * C::kStages;        // [2]
    r.p_full = r.s_full + 2;                  // [2]
    r.o_full = r.s_full + 4;
    r.drain = r.s_full + 5;
    r.a_tm = r.s_full + 6;
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

// A row warp's wait: lane 0 polls the barrier and shares the outcome; the
// warp-synchronous exchange orders the other lanes' later accesses after the
// completed phase (the row warps arrive once per warp for the same reason:
// 256 pollers and arrivals per step would contend with the tensor cores'
// shared-memory reads).
__device__ __forceinline__ bool row_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         int *err_word)
{
    int ok = 1;
    if ((threadIdx.x & 31) == 0)
        ok = ptx::mbar_wait(bar, parity, abort, err_word) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Shared set-up of both kernels: barriers, tensor memory, tensor-map prefetch.
// kv_full counts `kv_arrivals` arrivals (in the dK/dV kernel all lanes of the
// load warp arrive: they stage the statistics with the tiles).
template <int D>
__device__ __forceinline__ uint32_t setup(const BwdParams &p, const Bars &bar,
                                          uint32_t kv_arrivals, volatile int *abort_flag,
                                          uint32_t *tmem_slot)
{
    using C = Cfg<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar.a_full, 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bar.kv_full[s], kv_arrivals);
            ptx::mbar_init(&bar.kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bar.s_full[b], 1);
            ptx::mbar_init(&bar.p_full[b], kRowWarps);   // one arrival per row warp
        }
        ptx::mbar_init(bar.o_full, 1);
        ptx::mbar_init(bar.drain, 1);
        ptx::mbar_init(bar.a_tm, kRowWarps);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        ptx::prefetch_tmap(&p.tm_a0);
        ptx::prefetch_tmap(&p.tm_a1);
        ptx::prefetch_tmap(&p.tm_s0);
        ptx::prefetch_tmap(&p.tm_s1);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
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

// Columns [32 c_begin, 32 c_end) of row `r` of a 128-row accumulator (32-bit
// TMEM columns from t_acc) scaled by `mul`, written as bf16 to dst (the row's
// first element).
__device__ __forceinline__ void store_row(uint32_t t_acc, float mul, __nv_bfloat16 *dst, bool ok,
                                          int c_begin, int c_end)
{
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
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

// Shared-memory descriptor offsets of the K step kk (16 bf16) in a K-major
// 128B-swizzled tile whose 64-column chunks are `chunk_bytes` apart.
__device__ __forceinline__ uint64_t kmajor_off(int kk, uint32_t chunk_bytes)
{
    return uint64_t(((kk >> 2) * chunk_bytes + (kk & 3) * 32) >> 4);
}

// =============================================================================
// dQ (and D) -- one CTA per (sequence, head, query tile), heaviest tiles first
// =============================================================================
// Geometry of the dQ kernel: 128-key steps with S and dP single-buffered in
// TMEM -- S in columns [0, 128), dP in [128, 256) (dS packed into its first
// half per thread), dQ in [256, 256 + D), Q and dO as bf16 A operands after it.
// The MMA warp issues, per step j: S_{j+1} as soon as the rows have read S_j,
// dQ += dS_j K_j once they have stored dS_j, then dP_{j+1}; so the tensor
// pipe runs S_{j+1} while the rows finish dS_j, and only dQ_j waits for them.
// The ring holds K_j and V_j (128 rows each) in three stages: two of their
// own and, once the prologue has copied Q and dO into TMEM and formed D, the
// region that held the resident Q and dO tiles.
template <int D>
struct CfgQ {
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kTileBytes = BT * D * 2;       // one 128-row bf16 tile
    static constexpr uint32_t kStageBytes = 2 * kTileBytes;  // K_j, V_j
    static constexpr int kStages = 3;                         // stage 2 = the Q / dO region
    static constexpr uint32_t kOffRes = 0;
    static constexpr uint32_t kOffRing = 2 * kTileBytes;
    static constexpr uint32_t kOffXch = kOffRing + 2 * kStageBytes;   // 128 D_i values
    static constexpr uint32_t kOffBar = kOffXch + BT * 4;
    // a_full, kv_full[3], kv_empty[3], s_full, dp_full, s_free, p_full, o_full,
    // drain, a_tm, res_free
    static constexpr int kBars = 1 + 2 * kStages + 8;
    static constexpr uint32_t kSmemBytes = kOffBar + 8 * kBars + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static __device__ __forceinline__ uint32_t stage_off(int s)
    {
        return s == 2 ? kOffRes : kOffRing + uint32_t(s) * kStageBytes;
    }
};
constexpr uint32_t kQColS = 0, kQColDP = 128;   // dQ kernel: S; dP, then dS packed
constexpr int kQCols = 64;                      // columns of a step per row thread

template <int D, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
    using C = CfgQ<D>;
    // Q and dO as bf16 pairs in TMEM after the dQ accumulator (D / 2 columns
    // each): the A operands of S = Q K^T and dP = dO V^T
    constexpr uint32_t kColQA = kColAcc + D;
    static_assert(kColQA + D <= kTmemCols, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *a_full = bars, *kv_full = bars + 1, *kv_empty = bars + 1 + C::kStages;
    uint64_t *s_full = bars + 1 + 2 * C::kStages, *dp_full = s_full + 1, *s_free = s_full + 2,
             *p_full = s_full + 3, *o_full = s_full + 4, *drain = s_full + 5, *a_tm = s_full + 6,
             *res_free = s_full + 7;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + 8 * C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // work item (sequence, head, query tile), the heaviest query tiles first
    // within each group of (sequence, head) pairs (see bwd_head_groups)
    const int bh_count = p.B * p.H;
    int qt, bh;
    if (p.head_groups <= 1) {
        qt = p.n_tiles - 1 - int(blockIdx.x) / bh_count;
        bh = int(blockIdx.x) % bh_count;
    } else {
        const int gsz = bh_count / p.head_groups;
        const int grp = int(blockIdx.x) / (p.n_tiles * gsz);
        const int in_grp = int(blockIdx.x) - grp * (p.n_tiles * gsz);
        qt = p.n_tiles - 1 - in_grp / gsz;
        bh = grp * gsz + in_grp % gsz;
    }
    const int b = bh / p.H, h = bh % p.H;
    SeqRows sq;
    if (!seq_rows<PACKED>(p, b, h, sq) || qt * BT >= sq.L)
        return;                                     // whole CTA: nothing to do
    const int64_t row0 = sq.row0;                   // first row of the sequence
    const int L = sq.L;
    const int n_tiles = (L + BT - 1) / BT;
    // 128-key steps this query tile sees (at least one)
    const int n_kv = p.causal ? min(qt + 1, n_tiles) : n_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(a_full, 1);
        for (int st = 0; st < C::kStages; ++st) {
            ptx::mbar_init(&kv_full[st], 1);
            ptx::mbar_init(&kv_empty[st], 1);
        }
        ptx::mbar_init(s_full, 1);
        ptx::mbar_init(dp_full, 1);
        ptx::mbar_init(s_free, kRowWarps);
        ptx::mbar_init(p_full, kRowWarps);
        ptx::mbar_init(o_full, 1);
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(a_tm, kRowWarps);
        ptx::mbar_init(res_free, kRowWarps);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        ptx::prefetch_tmap(&p.tm_a0);
        ptx::prefetch_tmap(&p.tm_a1);
        ptx::prefetch_tmap(&p.tm_s0);
        ptx::prefetch_tmap(&p.tm_s1);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool aborted = false;
    uint8_t *tile_q = smem + C::kOffRes, *tile_do = tile_q + C::kTileBytes;

    if (warp == kWarpLoad) {
        // ======================= TMA producer ==============================
        if (lane == 0) {
            int last_phase[C::kStages];
            for (int st = 0; st < C::kStages; ++st)
                last_phase[st] = -1;
            ptx::mbar_arrive_expect_tx(a_full, 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                ptx::tma_load_3d(tile_q + c * kResChunkBytes, &p.tm_a0, a_full, c * 64, h,
                                 int(row0 + int64_t(qt) * BT));
                ptx::tma_load_3d(tile_do + c * kResChunkBytes, &p.tm_a1, a_full, c * 64, h,
                                 int(row0 + int64_t(qt) * BT));
            }
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < n_kv; ++j) {
                if (!ptx::mbar_wait(&kv_empty[stage], phase ^ 1u, abort_flag, p.err_word))
                    break;
                // stage 2 is the Q / dO region: free once the rows are done with it
                if (j == 2 && !ptx::mbar_wait(res_free, 0, abort_flag, p.err_word))
                    break;
                uint8_t *dst = smem + C::stage_off(stage);
                const int row = int(row0 + int64_t(j) * BT);
                ptx::mbar_arrive_expect_tx(&kv_full[stage], C::kStageBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    ptx::tma_load_3d(dst + c * kResChunkBytes, &p.tm_s0, &kv_full[stage], c * 64,
                                     h, row);
                    ptx::tma_load_3d(dst + C::kTileBytes + c * kResChunkBytes, &p.tm_s1,
                                     &kv_full[stage], c * 64, h, row);
                }
                if (j + C::kStages < n_kv)
                    for (int c = 0; c < C::kChunks; ++c) {
                        ptx::tma_prefetch_3d(&p.tm_s0, c * 64, h, row + C::kStages * BT);
                        ptx::tma_prefetch_3d(&p.tm_s1, c * 64, h, row + C::kStages * BT);
                    }
                last_phase[stage] = int(phase);
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (*abort_flag) {
                drain_wait(a_full, 0);
                for (int st = 0; st < C::kStages; ++st)
                    if (last_phase[st] >= 0)
                        drain_wait(&kv_full[st], uint32_t(last_phase[st]));
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer (whole warp) =====================
        constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BT, BT, false);   // N = 128 keys
        constexpr uint32_t idesc_q = ptx::idesc_bf16_f32(BT, D, true);     // B MN-major
        constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
        constexpr uint64_t desc_mnmajor = ptx::smem_desc_base(kResChunkBytes, 1024);
        // S = Q K^T into columns [0, 128) (A = Q from TMEM)
        auto issue_s = [&](uint32_t kaddr) {
            const uint64_t dk = ptx::smem_desc(desc_kmajor, kaddr);
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ts(tmem + kQColS, tmem + kColQA + 8 * kk,
                                dk + kmajor_off(kk, kResChunkBytes), idesc_s, kk > 0 ? 1u : 0u);
                ptx::mma_commit(s_full);
            }
            __syncwarp();
        };
        // dP = dO V^T into columns [128, 256) (A = dO from TMEM)
        auto issue_dp = [&](uint32_t vaddr) {
            const uint64_t dv = ptx::smem_desc(desc_kmajor, vaddr);
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ts(tmem + kQColDP, tmem + kColQA + D / 2 + 8 * kk,
                                dv + kmajor_off(kk, kResChunkBytes), idesc_s, kk > 0 ? 1u : 0u);
                ptx::mma_commit(dp_full);
            }
            __syncwarp();
        };
        const uint32_t smem_base = ptx::smem_u32(smem);
        do {
            if (!ptx::mbar_wait_warp(a_tm, 0, abort_flag, p.err_word) ||
                !ptx::mbar_wait_warp(&kv_full[0], 0, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            issue_s(smem_base + C::stage_off(0));
            issue_dp(smem_base + C::stage_off(0) + C::kTileBytes);
            int cur = 0;                               // ring stage of step j
            int nxt = 1;
            uint32_t nxt_phase = 0;                    // phase of step j + 1's stage
            for (int j = 0; j < n_kv; ++j) {
                const bool more = j + 1 < n_kv;
                if (more) {
                    // S_{j+1} overwrites S_j once every row has read it
                    if (!ptx::mbar_wait_warp(s_free, uint32_t(j) & 1u, abort_flag, p.err_word) ||
                        !ptx::mbar_wait_warp(&kv_full[nxt], nxt_phase, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    issue_s(smem_base + C::stage_off(nxt));
                }
                // dQ += dS_j K_j   (dS: bf16 packed in the first half of each
                // row thread's 64 dP columns; K_j an MN-major operand)
                if (!ptx::mbar_wait_warp(p_full, uint32_t(j) & 1u, abort_flag, p.err_word)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint64_t dkn = ptx::smem_desc(desc_mnmajor, smem_base + C::stage_off(cur));
                if (ptx::elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc,
                                    tmem + kQColDP + uint32_t(kQCols * (kk >> 2) + 8 * (kk & 3)),
                                    dkn + uint64_t((kk * 16 * 128) >> 4), idesc_q,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(&kv_empty[cur]);
                }
                __syncwarp();
                // dP_{j+1} overwrites dS_j after the dQ product has read it
                if (more)
                    issue_dp(smem_base + C::stage_off(nxt) + C::kTileBytes);
                cur = nxt;
                if (++nxt == C::kStages) {
                    nxt = 0;
                    nxt_phase ^= 1u;
                }
            }
        } while (false);
        if (ptx::elect_one()) {
            if (!aborted)
                ptx::mma_commit(o_full);
            ptx::mma_commit(drain);
            drain_wait(drain, 0);
        }
        __syncwarp();
    } else {
        // ======================= query rows ================================
        const int r = (warp & 3) * 32 + lane;        // query row in the tile = TMEM lane
        const int g = warp >> 2;                     // column group
        const int i = qt * BT + r;
        const bool row_ok = i < L;
        const uint32_t lane_bits = uint32_t((warp & 3) * 32) << 16;
        const int64_t stat = sq.stat0 + i;
        // D_i = dO_i . O_i (fp32), computed by the row warps together: a warp
        // takes 16 rows, D / 8 lanes per row, each lane 8 elements: O from
        // global memory (whole rows per load instruction), dO from the
        // resident shared-memory tile (128-byte swizzle: 16-byte unit u of row
        // r sits at unit u ^ (r % 8) of the row's 128 bytes in its 64-column
        // chunk).  The lanes of a row reduce with shuffles; the sums meet the
        // row threads in shared memory.
        constexpr int kLanesPerRow = D / 8, kRowsPerInst = 32 / kLanesPerRow;
        constexpr int kRowsPerWarp = BT / kRowWarps;          // 16
        float *xch = reinterpret_cast<float *>(smem + C::kOffXch);   // 128 sums
        {
            const int sub = lane / kLanesPerRow, lr = lane % kLanesPerRow;
            uint4 ov[kRowsPerWarp / kRowsPerInst];
#pragma unroll
            for (int k = 0; k < kRowsPerWarp / kRowsPerInst; ++k) {
                const int rr = warp * kRowsPerWarp + k * kRowsPerInst + sub;
                const int qi = qt * BT + rr;
                ov[k] = qi < L ? *reinterpret_cast<const uint4 *>(
                                       p.O + ((row0 + qi) * p.H + h) * D + lr * 8)
                                 : make_uint4(0, 0, 0, 0);
            }
            const bool a_ok = row_wait(a_full, 0, abort_flag, p.err_word);
            if (a_ok) {
                // this thread's half of row r of Q and of dO into TMEM, as the
                // bf16 pairs of the S and dP products' A operands
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint8_t *tile = t == 0 ? tile_q : tile_do;
                    uint32_t w[D / 4];
#pragma unroll
                    for (int ul = 0; ul < D / 16; ++ul) {
                        const int e0 = g * (D / 2) + ul * 8;          // first element
                        const int u = (e0 & 63) >> 3;
                        const uint4 v = *reinterpret_cast<const uint4 *>(
                            tile + (e0 >> 6) * kResChunkBytes + r * 128 + ((u ^ (r & 7)) << 4));
                        w[4 * ul + 0] = v.x;
                        w[4 * ul + 1] = v.y;
                        w[4 * ul + 2] = v.z;
                        w[4 * ul + 3] = v.w;
                    }
                    const uint32_t dst =
                        tmem + lane_bits + kColQA + uint32_t(t * (D / 2) + g * (D / 4));
                    if constexpr (D == 128)
                        ptx::tmem_st32(dst, w);
                    else
                        ptx::tmem_st16(dst, w);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(a_tm);
            }
#pragma unroll
            for (int k = 0; k < kRowsPerWarp / kRowsPerInst; ++k) {
                const int rr = warp * kRowsPerWarp + k * kRowsPerInst + sub;
                const int u = lr & 7, chunk = lr >> 3;
                const uint4 gv = a_ok ? *reinterpret_cast<const uint4 *>(
                                            tile_do + chunk * kResChunkBytes + rr * 128 +
                                            ((u ^ (rr & 7)) << 4))
                                      : make_uint4(0, 0, 0, 0);
                const uint32_t ow[4] = {ov[k].x, ov[k].y, ov[k].z, ov[k].w};
                const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 of =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ow[e]));
                    const float2 gf =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gw[e]));
                    part = fmaf(of.x, gf.x, part);
                    part = fmaf(of.y, gf.y, part);
                }
#pragma unroll
                for (int o = kLanesPerRow / 2; o > 0; o >>= 1)
                    part += __shfl_xor_sync(0xffffffffu, part, o);
                if (lr == 0)
                    xch[rr] = part;
            }
            // this warp has finished with the Q / dO region (ring stage 2)
            __syncwarp();
            if (a_ok && lane == 0)
                ptx::mbar_arrive(res_free);
        }
        const float lse_raw = row_ok ? p.lse[stat] : 0.f;
        asm volatile("bar.sync 1, %0;" ::"n"(BT * G) : "memory");   // the row threads
        const float Di = xch[r];
        if (g == 0 && row_ok)
            p.D[stat] = Di;
        const float lse2 = lse_raw * kLog2e;
        const float sl = p.scale_log2;
        const int col0 = g * kQCols;
        const uint32_t tS = tmem + lane_bits + kQColS + uint32_t(col0);
        const uint32_t tDP = tmem + lane_bits + kQColDP + uint32_t(col0);

        for (int j = 0; j < n_kv; ++j) {
            const uint32_t par = uint32_t(j) & 1u;
            if (!row_wait(s_full, par, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            // last visible column of this key tile for row i (causal diagonal,
            // end of the sequence); rows past the end see nothing
            int lim = BT - 1;
            if (p.causal && i - j * BT < lim)
                lim = i - j * BT;
            if (L - 1 - j * BT < lim)
                lim = L - 1 - j * BT;
            if (!row_ok)
                lim = -1;
            float pr[kQCols];
            {
                uint32_t sv0[32], sv1[32];
                ptx::tmem_ld32(tS, sv0);
                ptx::tmem_ld32(tS + 32, sv1);
                ptx::tmem_wait_ld();
                // S is read: the MMA warp may overwrite it with the next step's
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(s_free);
                // masked entries get exponent -inf: exp2 gives 0, no branch
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const int c0 = col0 + k, c1 = col0 + 32 + k;
                    pr[k] = ptx::ex2(c0 <= lim ? fmaf(__uint_as_float(sv0[k]), sl, -lse2)
                                               : -INFINITY);
                    pr[32 + k] = ptx::ex2(c1 <= lim ? fmaf(__uint_as_float(sv1[k]), sl, -lse2)
                                                    : -INFINITY);
                }
            }
            if (!row_wait(dp_full, par, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            uint32_t pk[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t dv[32];
                ptx::tmem_ld32(tDP + 32 * half, dv);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float d0 = pr[32 * half + 2 * e] * (__uint_as_float(dv[2 * e]) - Di);
                    const float d1 =
                        pr[32 * half + 2 * e + 1] * (__uint_as_float(dv[2 * e + 1]) - Di);
                    pk[16 * half + e] = ptx::pack_bf16x2(d0, d1);
                }
            }
            ptx::tmem_st32(tDP, pk);                  // dS of this row's 64 keys, packed
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(p_full);
        }
        // the two groups store half of each row's dQ each
        if (!aborted && ptx::mbar_wait(o_full, 0, abort_flag, p.err_word)) {
            ptx::tc_fence_after_sync();
            store_row(tmem + lane_bits + kColAcc, p.scale, p.dQ + ((row0 + i) * p.H + h) * D,
                      row_ok, g * (D / 64), (g + 1) * (D / 64));
        }
    }
    teardown<D>(tmem);
}

// =============================================================================
// dK, dV -- one CTA per (sequence, head, key tile), heaviest tiles first
// =============================================================================
template <int D, bool PACKED>
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

    // work item (sequence, head, key tile): low key tiles (the most query
    // steps when causal) first within each group of (sequence, head) pairs
    const int bh_count = p.B * p.H;
    int kt, bh;
    if (p.head_groups <= 1) {
        kt = int(blockIdx.x) / bh_count;
        bh = int(blockIdx.x) % bh_count;
    } else {
        const int gsz = bh_count / p.head_groups;
        const int grp = int(blockIdx.x) / (p.n_tiles * gsz);
        const int in_grp = int(blockIdx.x) - grp * (p.n_tiles * gsz);
        kt = in_grp / gsz;
        bh = grp * gsz + in_grp % gsz;
    }
    const int b = bh / p.H, h = bh % p.H;
    SeqRows sq;
    if (!seq_rows<PACKED>(p, b, h, sq) || kt * BT >= sq.L)
        return;                                      // whole CTA: nothing to do
    const int64_t row0 = sq.row0;
    const int L = sq.L;
    const int n_sub = (L + BS - 1) / BS;
    // first query sub-tile that sees the keys; at least one sub-tile follows
    const int i0 = p.causal ? 2 * kt : 0;
    const int n_q = n_sub - i0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t tmem = setup<D>(p, bar, 32u, abort_flag, tmem_slot);
    bool aborted = false;
    uint8_t *tile_k = smem + C::kOffA0, *tile_v = smem + C::kOffA1;
    uint8_t *ring = smem + C::kOffRing;
    float *stats = reinterpret_cast<float *>(smem + C::kOffStat);   // slot x (lse2, D) x 64

    if (warp == kWarpLoad) {
        // ======================= TMA producer (whole warp) ===================
        // Ring stage of step s (i = i0 + s): Q_i then dO_i; the warp's lanes
        // also stage the sub-tile's log2 logsumexp and D in the stage's slot.
        int last_phase[C::kStages];
        for (int s = 0; s < C::kStages; ++s)
            last_phase[s] = -1;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar.a_full, 2 * C::kResBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                ptx::tma_load_3d(tile_k + c * kResChunkBytes, &p.tm_a0, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
                ptx::tma_load_3d(tile_v + c * kResChunkBytes, &p.tm_a1, bar.a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
            }
        }
        int stage = 0;
        uint32_t phase = 0;
        const int64_t stat0 = sq.stat0;
        // Launched as a programmatic dependent of the dQ kernel: K and V
        // (inputs) are requested above; D is that kernel's output, and every
        // lane of this warp loads it, so all of them wait for its completion.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        for (int s = 0; s < n_q; ++s) {
            const int i = i0 + s;
            // the step's statistics: global loads in flight during the slot wait
            float ls[BS / 32], ds[BS / 32];
#pragma unroll
            for (int u = 0; u < BS / 32; ++u) {
                const int q = i * BS + lane * (BS / 32) + u;
                const bool v = q < L;
                ls[u] = v ? p.lse[stat0 + q] : 0.f;
                ds[u] = v ? p.D[stat0 + q] : 0.f;
            }
            int ok = 1;
            if (lane == 0)
                ok = ptx::mbar_wait(&bar.kv_empty[stage], phase ^ 1u, abort_flag, p.err_word) ? 1
                                                                                             : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0))
                break;
            if (lane == 0) {
                uint8_t *dst = ring + stage * C::kStageBytes;
                const int row = int(row0 + int64_t(i) * BS);
                ptx::mbar_expect_tx(&bar.kv_full[stage], C::kStageBytes);
                for (int c = 0; c < C::kChunks; ++c) {
                    ptx::tma_load_3d(dst + c * kSubChunkBytes, &p.tm_s0, &bar.kv_full[stage],
                                     c * 64, h, row);
                    ptx::tma_load_3d(dst + C::kSubBytes + c * kSubChunkBytes, &p.tm_s1,
                                     &bar.kv_full[stage], c * 64, h, row);
                }
                if (i + kL2Ahead < n_sub)
                    for (int c = 0; c < C::kChunks; ++c) {
                        ptx::tma_prefetch_3d(&p.tm_s0, c * 64, h, row + kL2Ahead * BS);
                        ptx::tma_prefetch_3d(&p.tm_s1, c * 64, h, row + kL2Ahead * BS);
                    }
                last_phase[stage] = int(phase);
            }
            float *slot = stats + stage * (2 * BS);
#pragma unroll
            for (int u = 0; u < BS / 32; ++u) {
                slot[lane * (BS / 32) + u] = ls[u] * kLog2e;
                slot[BS + lane * (BS / 32) + u] = ds[u];
            }
            ptx::mbar_arrive(&bar.kv_full[stage]);       // all 32 lanes, after their writes
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (lane == 0 && *abort_flag) {
            drain_wait(bar.a_full, 0);
            for (int s = 0; s < C::kStages; ++s)
                if (last_phase[s] >= 0)
                    drain_wait(&bar.kv_full[s], uint32_t(last_phase[s]));
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer (whole warp) =====================
        // Order: S^T_0, dP^T_0; then per step s: S^T_{s+1}, dP^T_{s+1} (other
        // buffer), wait for P^T_s and dS^T_s, dV += P^T_s dO_s, dK += dS^T_s Q_s.
        // The warp runs the loop converged; one elected lane issues.
        constexpr uint32_t idesc_ss = ptx::idesc_bf16_f32(BT, BS, false);
        constexpr uint32_t idesc_ts = ptx::idesc_bf16_f32(BT, D, true);
        constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
        constexpr uint64_t desc_mnmajor = ptx::smem_desc_base(kSubChunkBytes, 1024);
        const uint64_t dk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_k));
        const uint64_t dvk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_v));
        const uint32_t ring_addr = ptx::smem_u32(ring);
        int stage = 0;
        uint32_t phase = 0;
        int st0 = 0, st1 = 0;                       // step's ring stage, per buffer
        // S^T_s = K Q_s^T and dP^T_s = V dO_s^T into buffer s & 1
        auto issue_s = [&](int s) -> bool {
            if (!ptx::mbar_wait_warp(&bar.kv_full[stage], phase, abort_flag, p.err_word))
                return false;
            (s & 1 ? st1 : st0) = stage;
            const uint32_t qaddr = ring_addr + stage * C::kStageBytes;
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
            ptx::tc_fence_after_sync();
            const uint64_t dq = ptx::smem_desc(desc_kmajor, qaddr);
            const uint64_t ddo = ptx::smem_desc(desc_kmajor, qaddr + C::kSubBytes);
            const uint32_t buf = tmem + uint32_t(s & 1) * kColBuf;
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(buf, dk + kmajor_off(kk, kResChunkBytes),
                                dq + kmajor_off(kk, kSubChunkBytes), idesc_ss, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(buf + kColDP, dvk + kmajor_off(kk, kResChunkBytes),
                                ddo + kmajor_off(kk, kSubChunkBytes), idesc_ss, kk > 0 ? 1u : 0u);
                ptx::mma_commit(&bar.s_full[s & 1]);
            }
            __syncwarp();
            return true;
        };
        do {
            if (!ptx::mbar_wait_warp(bar.a_full, 0, abort_flag, p.err_word) || !issue_s(0)) {
                aborted = true;
                break;
            }
            for (int s = 0; s < n_q; ++s) {
                if (s + 1 < n_q && !issue_s(s + 1)) {
                    aborted = true;
                    break;
                }
                // dV += P^T_s dO_s,  dK += dS^T_s Q_s
                if (!ptx::mbar_wait_warp(&bar.p_full[s & 1], uint32_t(s >> 1) & 1u, abort_flag,
                                         p.err_word)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const int st = (s & 1) ? st1 : st0;
                const uint32_t qaddr = ring_addr + st * C::kStageBytes;
                const uint64_t dq_mn = ptx::smem_desc(desc_mnmajor, qaddr);
                const uint64_t ddo_mn = ptx::smem_desc(desc_mnmajor, qaddr + C::kSubBytes);
                const uint32_t a_tm = tmem + uint32_t(s & 1) * kColBuf;
                if (ptx::elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc, a_tm + packed_col(kk),
                                    ddo_mn + uint64_t((kk * 16 * 128) >> 4), idesc_ts,
                                    (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        ptx::mma_ts(tmem + kColAcc + D, a_tm + kColDP + packed_col(kk),
                                    dq_mn + uint64_t((kk * 16 * 128) >> 4), idesc_ts,
                                    (s > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(&bar.kv_empty[st]);
                }
                __syncwarp();
            }
        } while (false);
        if (ptx::elect_one()) {
            if (!aborted)
                ptx::mma_commit(bar.o_full);
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
        const float sl = p.scale_log2;
        const int col0 = g * kColsPerThread;
        for (int s = 0; s < n_q; ++s) {
            const int i = i0 + s;
            // the statistics arrive with the step's ring stage; they are read
            // into registers before the wait for S^T_s
            const int st = s % C::kStages;
            if (!row_wait(&bar.kv_full[st], uint32_t(s / C::kStages) & 1u, abort_flag,
                                p.err_word)) {
                aborted = true;
                break;
            }
            float lv[32], dd[32];
            {
                const float *lse2s = stats + st * (2 * BS) + col0;
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 l4 = *reinterpret_cast<const float4 *>(lse2s + 4 * e4);
                    const float4 d4 = *reinterpret_cast<const float4 *>(lse2s + BS + 4 * e4);
                    lv[4 * e4] = l4.x;
                    lv[4 * e4 + 1] = l4.y;
                    lv[4 * e4 + 2] = l4.z;
                    lv[4 * e4 + 3] = l4.w;
                    dd[4 * e4] = d4.x;
                    dd[4 * e4 + 1] = d4.y;
                    dd[4 * e4 + 2] = d4.z;
                    dd[4 * e4 + 3] = d4.w;
                }
            }
            if (!row_wait(&bar.s_full[s & 1], uint32_t(s >> 1) & 1u, abort_flag,
                                p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            // visible columns [lo, hi]: causal keeps queries >= the key; the
            // sequence ends at N
            const int lo = p.causal ? k - i * BS : 0;
            int hi = L - 1 - i * BS;
            if (hi > BS - 1)
                hi = BS - 1;
            const uint32_t tS = tmem + lane_bits + uint32_t(s & 1) * kColBuf + col0;
            uint32_t sv[32], dv[32], pk[16], dk[16];
            ptx::tmem_ld32(tS, sv);
            ptx::tmem_ld32(tS + kColDP, dv);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                float pv[2], ds[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = 2 * e2 + u;
                    const int c = col0 + e;
                    const float x = __uint_as_float(sv[e]);
                    const float y = __uint_as_float(dv[e]);
                    // masked entries get exponent -inf: exp2 gives 0, no branch
                    pv[u] = ptx::ex2((c >= lo && c <= hi) ? fmaf(x, sl, -lv[e]) : -INFINITY);
                    ds[u] = pv[u] * (y - dd[e]);
                }
                pk[e2] = ptx::pack_bf16x2(pv[0], pv[1]);
                dk[e2] = ptx::pack_bf16x2(ds[0], ds[1]);
            }
            ptx::tmem_st16(tS, pk);                   // P^T of this block, packed
            ptx::tmem_st16(tS + kColDP, dk);          // dS^T of this block, packed
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&bar.p_full[s & 1]);
        }
        if (!aborted && ptx::mbar_wait(bar.o_full, 0, abort_flag, p.err_word)) {
            ptx::tc_fence_after_sync();
            const bool key_ok = k < L;
            // group 0 writes dV, group 1 writes dK
            if (g == 0)
                store_row(tmem + lane_bits + kColAcc, 1.f, p.dV + ((row0 + k) * p.H + h) * D,
                          key_ok, 0, D / 32);
            else
                store_row(tmem + lane_bits + kColAcc + D, p.scale,
                          p.dK + ((row0 + k) * p.H + h) * D, key_ok, 0, D / 32);
        }
    }
    teardown<D>(tmem);
}

// =============================================================================
// One-pass backward (d = 128, dense or packed): dK, dV and each key tile's
// share of dQ
// =============================================================================
// One CTA per (sequence, head, 128-key tile), as the dK/dV kernel, that also
// forms dQ^T_s = K^T dS^T_s for each 64-query sub-step and adds it into an
// fp32 accumulator ([B*H, n_pad, d]; packed: [H, total + 64, d]) in global
// memory with atomic adds: the
// contributions of the key tiles are summed in L2 ("少搬一趟…" §3.3: the
// column blocks' dQ shares summed with atomic adds; §5.6). The order of those
// adds varies from run to run, so dQ's rounding may too; dK and dV do not.
// TMEM: S^T in two buffers [0, 64), [64, 128) (P^T packed into them); dP^T
// single-buffered in [128, 192); dQ^T in [192, 256) (lanes = head-dim index,
// columns = queries); dV in [256, 384); dK in [384, 512).
// Shared memory: K and V resident; a 3-stage ring of (Q_s, dO_s); dS^T in two
// 16 KB buffers (row = key, 64 queries = 128 bytes, 128-byte swizzle), which
// is both the K-major A operand of dK += dS^T Q_s and the MN-major B operand
// of dQ^T = K^T dS^T.
template <int D_>
struct CfgF {
    static constexpr int D = D_;
    static constexpr int kChunks = D / 64;
    static constexpr uint32_t kResBytes = BT * D * 2;
    static constexpr uint32_t kSubBytes = BS * D * 2;
    static constexpr int kStages = 3;
    static constexpr uint32_t kStageBytes = 2 * kSubBytes;
    static constexpr uint32_t kDsBytes = BT * BS * 2;
    // K^T is the A operand of dQ^T with M = 128 head-dim rows in two 64-row
    // blocks 16 KB apart: at d = 128 the second block is K's second chunk; at
    // d = 64 it is a zero tile placed there, so the operand and its descriptor
    // are the same for both head dims (the padded rows of dQ^T are zeros)
    static constexpr uint32_t kOffA0 = 0;
    static constexpr uint32_t kOffZero = kResChunkBytes;      // d = 64 only
    static constexpr uint32_t kOffA1 = 2 * kResChunkBytes;    // V
    static constexpr uint32_t kOffRing = kOffA1 + kResBytes;
    static constexpr uint32_t kOffDs = kOffRing + kStages * kStageBytes;
    static constexpr uint32_t kOffStat = kOffDs + 2 * kDsBytes;
    static constexpr uint32_t kStatBytes = kStages * 2 * BS * 4;   // (lse log2 e, D) pairs
    static constexpr uint32_t kOffBar = kOffStat + kStatBytes;
    // a_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], dp_read, dq_full,
    // dq_free, o_full, drain, never (nothing arrives: failure-detection test)
    static constexpr int kBars = 1 + 2 * kStages + 10;
    static constexpr uint32_t kSmemBytes = kOffBar + 8 * kBars + 16 + 1024;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};
constexpr uint32_t kFColDP = 128, kFColDQ = 192, kFColDV = 256;   // dK from 256 + d

template <int D, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_fused_kernel(const __grid_constant__ BwdParams p)
{
    using C = CfgF<D>;
    constexpr uint32_t kFColDK = kFColDV + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    uint64_t *a_full = bars, *kv_full = bars + 1, *kv_empty = bars + 1 + C::kStages;
    uint64_t *s_full = bars + 1 + 2 * C::kStages;          // [2]
    uint64_t *p_full = s_full + 2;                          // [2]
    uint64_t *dp_read = s_full + 4, *dq_full = s_full + 5, *dq_free = s_full + 6,
             *o_full = s_full + 7, *drain = s_full + 8, *never = s_full + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffBar + 8 * C::kBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // work item (sequence, head, key tile): low key tiles (the most query
    // steps when causal) first within each group of (sequence, head) pairs;
    // the groups run one after another so that a group's Q, dO and dQ sums
    // stay in L2
    const int bh_count = p.B * p.H;
    int kt, bh;
    if (p.head_groups <= 1) {
        kt = int(blockIdx.x) / bh_count;
        bh = int(blockIdx.x) % bh_count;
    } else {
        const int gsz = bh_count / p.head_groups;
        const int grp = int(blockIdx.x) / (p.n_tiles * gsz);
        const int in_grp = int(blockIdx.x) - grp * (p.n_tiles * gsz);
        kt = in_grp / gsz;
        bh = grp * gsz + in_grp % gsz;
    }
    const int b = bh / p.H, h = bh % p.H;
    SeqRows sq;
    if (!seq_rows<PACKED>(p, b, h, sq) || kt * BT >= sq.L)
        return;                                      // whole CTA: nothing to do
    const int64_t row0 = sq.row0;
    const int L = sq.L;
    const int n_sub = (L + BS - 1) / BS;
    const int i0 = p.causal ? 2 * kt : 0;            // first query sub-tile that sees the keys
    const int n_q = n_sub - i0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(a_full, 1);
        for (int st = 0; st < C::kStages; ++st) {
            ptx::mbar_init(&kv_full[st], 1);
            ptx::mbar_init(&kv_empty[st], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&s_full[i], 1);
            ptx::mbar_init(&p_full[i], kRowWarps);
        }
        ptx::mbar_init(dp_read, kRowWarps);
        ptx::mbar_init(dq_full, 1);
        ptx::mbar_init(dq_free, kRowWarps);
        ptx::mbar_init(o_full, 1);
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(never, 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kWarpMma) {
        ptx::tmem_alloc(tmem_slot, kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == kWarpLoad && lane == 0) {
        ptx::prefetch_tmap(&p.tm_a0);
        ptx::prefetch_tmap(&p.tm_a1);
        ptx::prefetch_tmap(&p.tm_s0);
        ptx::prefetch_tmap(&p.tm_s1);
    }
    if constexpr (D < 128) {
        // the zero rows of the K^T operand (see CfgF)
        for (int i = threadIdx.x; i < int(kResChunkBytes / 16); i += kThreads)
            reinterpret_cast<uint4 *>(smem + C::kOffZero)[i] = make_uint4(0, 0, 0, 0);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool aborted = false;
    uint8_t *tile_k = smem + C::kOffA0, *tile_v = smem + C::kOffA1;
    uint8_t *ring = smem + C::kOffRing;
    float *stats = reinterpret_cast<float *>(smem + C::kOffStat);   // slot x (lse2, D) x 64

    if (warp == kWarpLoad) {
        // ======================= TMA producer ==============================
        // Ring stage of step s: Q_s, dO_s and the sub-tile's 64 (lse log2 e,
        // D) pairs, all on the stage's barrier; one lane issues everything.
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(a_full, 2 * C::kResBytes);
            for (int c = 0; c < C::kChunks; ++c) {
                ptx::tma_load_3d(tile_k + c * kResChunkBytes, &p.tm_a0, a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
                ptx::tma_load_3d(tile_v + c * kResChunkBytes, &p.tm_a1, a_full, c * 64, h,
                                 int(row0 + int64_t(kt) * BT));
            }
            const int64_t stat_row = PACKED ? int64_t(h) * p.B + b : int64_t(bh);
            const float2 *stat_src = p.stat2 + stat_row * p.n_pad;
            // Launched as a programmatic dependent of the prep kernel: the
            // resident K, V (inputs) are requested above; the statistics and
            // the zeroed accumulator are that kernel's output, so the copies
            // below wait for it to complete.  Every other role reaches them
            // only through the ring barriers filled after this wait (the rows'
            // atomic adds follow their first kv_full wait).
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int issued = 0;
            for (int s = 0; s < n_q; ++s) {
                const int stage = s % C::kStages;
                const uint32_t phase = uint32_t(s / C::kStages) & 1u;
                if (!ptx::mbar_wait(&kv_empty[stage], phase ^ 1u, abort_flag, p.err_word))
                    break;
                const int i = i0 + s;
                uint8_t *dst = ring + stage * C::kStageBytes;
                const int row = int(row0 + int64_t(i) * BS);
                ptx::mbar_arrive_expect_tx(&kv_full[stage], C::kStageBytes + 2 * BS * 4);
                for (int c = 0; c < C::kChunks; ++c) {
                    ptx::tma_load_3d(dst + c * kSubChunkBytes, &p.tm_s0, &kv_full[stage], c * 64,
                                     h, row);
                    ptx::tma_load_3d(dst + C::kSubBytes + c * kSubChunkBytes, &p.tm_s1,
                                     &kv_full[stage], c * 64, h, row);
                }
                ptx::bulk_load(stats + stage * (2 * BS), stat_src + int64_t(i) * BS, 2 * BS * 4,
                               &kv_full[stage]);
                if (i + kL2Ahead < n_sub)
                    for (int c = 0; c < C::kChunks; ++c) {
                        ptx::tma_prefetch_3d(&p.tm_s0, c * 64, h, row + kL2Ahead * BS);
                        ptx::tma_prefetch_3d(&p.tm_s1, c * 64, h, row + kL2Ahead * BS);
                    }
                issued = s + 1;
            }
            // wait (bounded) for the copies in flight before the CTA ends: the
            // last step issued into each stage.  Done whether or not the flag
            // is up yet: a short test timeout can raise it after this point,
            // and without an abort these phases have completed or are about to.
            drain_wait(a_full, 0);
            for (int s = issued - C::kStages > 0 ? issued - C::kStages : 0; s < issued; ++s)
                drain_wait(&kv_full[s % C::kStages], uint32_t(s / C::kStages) & 1u);
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer (whole warp) =====================
        // Pipe order per step s: S^T_{s+1}, dP^T_{s+1} (once the rows have
        // read dP^T_s), dV += P^T_s dO_s, dK += dS^T_s Q_s, dQ^T_s = K^T dS^T_s
        // (once the rows have read dQ^T_{s-1}).  One elected lane issues.
        constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(BT, BS, false);
        constexpr uint32_t idesc_acc = ptx::idesc_bf16_f32(BT, D, true);          // B MN-major
        constexpr uint32_t idesc_dq = ptx::idesc_bf16_f32_mn(BT, BS, true, true); // both MN-major
        constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
        constexpr uint64_t desc_mn_sub = ptx::smem_desc_base(kSubChunkBytes, 1024);
        constexpr uint64_t desc_mn_res = ptx::smem_desc_base(kResChunkBytes, 1024);
        constexpr uint64_t desc_mn_ds = ptx::smem_desc_base(C::kDsBytes, 1024);
        const uint64_t dk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_k));
        const uint64_t dvk = ptx::smem_desc(desc_kmajor, ptx::smem_u32(tile_v));
        const uint64_t dkt = ptx::smem_desc(desc_mn_res, ptx::smem_u32(tile_k));   // K^T
        const uint32_t ring_addr = ptx::smem_u32(ring);
        const uint32_t ds_addr = ptx::smem_u32(smem + C::kOffDs);
        auto stage_addr = [&](int s) { return ring_addr + (s % C::kStages) * C::kStageBytes; };
        // S^T_s = K Q_s^T into buffer s & 1 (waits for the step's ring stage)
        auto issue_s = [&](int s) -> bool {
            if (!ptx::mbar_wait_warp(&kv_full[s % C::kStages], uint32_t(s / C::kStages) & 1u,
                                     abort_flag, p.err_word))
                return false;
            ptx::tc_fence_after_sync();
            const uint64_t dq = ptx::smem_desc(desc_kmajor, stage_addr(s));
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + uint32_t(s & 1) * BS, dk + kmajor_off(kk, kResChunkBytes),
                                dq + kmajor_off(kk, kSubChunkBytes), idesc_s, kk > 0 ? 1u : 0u);
            }
            __syncwarp();
            return true;
        };
        // dP^T_s = V dO_s^T into the dP^T columns; completes s_full[s & 1]
        auto issue_dp = [&](int s) {
            const uint64_t ddo = ptx::smem_desc(desc_kmajor, stage_addr(s) + C::kSubBytes);
            if (ptx::elect_one()) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    ptx::mma_ss(tmem + kFColDP, dvk + kmajor_off(kk, kResChunkBytes),
                                ddo + kmajor_off(kk, kSubChunkBytes), idesc_s, kk > 0 ? 1u : 0u);
                ptx::mma_commit(&s_full[s & 1]);
            }
            __syncwarp();
        };
        // Failure-detection test: a wait on a barrier that nothing arrives at
        // runs out after expire_wait_ns; it raises the error bit and the abort
        // flag, and the CTA winds down as after any timed-out wait.
        if (p.expire_wait_ns != 0u &&
            !__all_sync(0xffffffffu, ptx::mbar_wait_limited(never, 0, abort_flag, p.err_word,
                                                            p.expire_wait_ns)))
            aborted = true;
        do {
            if (aborted || !ptx::mbar_wait_warp(a_full, 0, abort_flag, p.err_word) ||
                !issue_s(0)) {
                aborted = true;
                break;
            }
            issue_dp(0);
            for (int s = 0; s < n_q; ++s) {
                if (s + 1 < n_q) {
                    if (!issue_s(s + 1) ||
                        !ptx::mbar_wait_warp(dp_read, uint32_t(s) & 1u, abort_flag, p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    issue_dp(s + 1);
                }
                if (!ptx::mbar_wait_warp(&p_full[s & 1], uint32_t(s >> 1) & 1u, abort_flag,
                                         p.err_word)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                const uint32_t qaddr = stage_addr(s);
                const uint64_t dq_mn = ptx::smem_desc(desc_mn_sub, qaddr);
                const uint64_t ddo_mn = ptx::smem_desc(desc_mn_sub, qaddr + C::kSubBytes);
                const uint32_t dsb = ds_addr + uint32_t(s & 1) * C::kDsBytes;
                const uint64_t ds_k = ptx::smem_desc(desc_kmajor, dsb);    // dS^T as A
                const uint64_t ds_mn = ptx::smem_desc(desc_mn_ds, dsb);    // dS^T as B
                const uint32_t a_tm = tmem + uint32_t(s & 1) * BS;
                if (ptx::elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        ptx::mma_ts(tmem + kFColDV, a_tm + packed_col(kk),
                                    ddo_mn + uint64_t((kk * 16 * 128) >> 4), idesc_acc,
                                    (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < BS / 16; ++kk)
                        ptx::mma_ss(tmem + kFColDK, ds_k + uint64_t((kk * 32) >> 4),
                                    dq_mn + uint64_t((kk * 16 * 128) >> 4), idesc_acc,
                                    (s > 0 || kk > 0) ? 1u : 0u);
                    ptx::mma_commit(&kv_empty[s % C::kStages]);
                }
                __syncwarp();
                if (s > 0 &&
                    !ptx::mbar_wait_warp(dq_free, uint32_t(s - 1) & 1u, abort_flag, p.err_word)) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                if (ptx::elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BT / 16; ++kk)
                        ptx::mma_ss(tmem + kFColDQ, dkt + uint64_t((kk * 16 * 128) >> 4),
                                    ds_mn + uint64_t((kk * 16 * 128) >> 4), idesc_dq,
                                    kk > 0 ? 1u : 0u);
                    ptx::mma_commit(dq_full);
                }
                __syncwarp();
            }
        } while (false);
        if (ptx::elect_one()) {
            if (!aborted)
                ptx::mma_commit(o_full);
            ptx::mma_commit(drain);
            drain_wait(drain, 0);
        }
        __syncwarp();
    } else {
        // ======================= key rows ==================================
        const int r = (warp & 3) * 32 + lane;        // key row = TMEM lane (= head-dim
                                                     // index of dQ^T)
        const int g = warp >> 2;                     // column group
        const int k = kt * BT + r;
        const uint32_t lane_bits = uint32_t((warp & 3) * 32) << 16;
        const float sl = p.scale_log2;
        const int col0 = g * kColsPerThread;
        // dQ^T of step t: load this thread's 32 queries of head-dim row r,
        // free the columns, and add them into the accumulator (a warp's 32
        // lanes hold one query's 32 consecutive head-dim entries: one 128-byte
        // row per atomic instruction).  Queries past the sequence's end add
        // zeros (their dS is 0), into rows that belong to no query of it.
        const int64_t acc_row0 = PACKED ? int64_t(h) * p.total_pad + row0 : int64_t(bh) * p.n_pad;
        // (at d = 64 the warps of lanes 64 .. 127 hold the zero rows: they
        // only keep the barrier protocol)
        const bool has_d = (warp & 3) * 32 < D;
        auto drain_dq = [&](int t) -> bool {
            if (!row_wait(dq_full, uint32_t(t) & 1u, abort_flag, p.err_word))
                return false;
            ptx::tc_fence_after_sync();
            if (has_d) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_bits + kFColDQ + col0, v);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(dq_free);
                float *dst = p.dq_acc + (acc_row0 + (i0 + t) * BS + col0) * D + r;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    ptx::red_add_f32(dst + c * D, __uint_as_float(v[c]));
            } else {
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(dq_free);
            }
            return true;
        };
        for (int s = 0; s < n_q; ++s) {
            const int i = i0 + s;
            const int st = s % C::kStages;
            if (!row_wait(&kv_full[st], uint32_t(s / C::kStages) & 1u, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            float lv[32], dd[32];
            {
                // (lse log2 e, D) pairs of the step's queries col0 .. col0 + 31
                const float4 *st4 =
                    reinterpret_cast<const float4 *>(stats + st * (2 * BS) + 2 * col0);
#pragma unroll
                for (int e2 = 0; e2 < 16; ++e2) {
                    const float4 v4 = st4[e2];
                    lv[2 * e2] = v4.x;
                    dd[2 * e2] = v4.y;
                    lv[2 * e2 + 1] = v4.z;
                    dd[2 * e2 + 1] = v4.w;
                }
            }
            if (!row_wait(&s_full[s & 1], uint32_t(s >> 1) & 1u, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            // visible columns [lo, hi]: causal keeps queries >= the key, the
            // sequence ends at L; a key row past the end (the next sequence's
            // K row in a dense batch) sees none, so it adds nothing to dQ
            const int lo = k >= L ? BS : (p.causal ? k - i * BS : 0);
            int hi = L - 1 - i * BS;
            if (hi > BS - 1)
                hi = BS - 1;
            const uint32_t tS = tmem + lane_bits + uint32_t(s & 1) * BS + col0;
            uint32_t sv[32], dv[32], pk[16], dk[16];
            ptx::tmem_ld32(tS, sv);
            ptx::tmem_ld32(tmem + lane_bits + kFColDP + col0, dv);
            ptx::tmem_wait_ld();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(dp_read);            // dP^T_{s+1} may overwrite the columns
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
                float pv[2], ds[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = 2 * e2 + u;
                    const int c = col0 + e;
                    const float x = __uint_as_float(sv[e]);
                    const float y = __uint_as_float(dv[e]);
                    pv[u] = ptx::ex2((c >= lo && c <= hi) ? fmaf(x, sl, -lv[e]) : -INFINITY);
                    ds[u] = pv[u] * (y - dd[e]);
                }
                pk[e2] = ptx::pack_bf16x2(pv[0], pv[1]);
                dk[e2] = ptx::pack_bf16x2(ds[0], ds[1]);
            }
            ptx::tmem_st16(tS, pk);                   // P^T of this block, packed
            // dS^T row r, queries [col0, col0 + 32): 16-byte units 4g .. 4g + 3
            uint8_t *dsrow = smem + C::kOffDs + (s & 1) * C::kDsBytes + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4 *>(dsrow + (((4 * g + j) ^ (r & 7)) << 4)) =
                    make_uint4(dk[4 * j], dk[4 * j + 1], dk[4 * j + 2], dk[4 * j + 3]);
            ptx::tmem_wait_st();
            ptx::fence_proxy_async_smem();            // dS^T -> the tensor cores
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(&p_full[s & 1]);
            if (s > 0 && !drain_dq(s - 1)) {
                aborted = true;
                break;
            }
        }
        if (!aborted && n_q > 0 && !drain_dq(n_q - 1))
            aborted = true;
        if (!aborted && ptx::mbar_wait(o_full, 0, abort_flag, p.err_word)) {
            ptx::tc_fence_after_sync();
            const bool key_ok = k < L;
            if (g == 0)
                store_row(tmem + lane_bits + kFColDV, 1.f, p.dV + ((row0 + k) * p.H + h) * D,
                          key_ok, 0, D / 32);
            else
                store_row(tmem + lane_bits + kFColDK, p.scale,
                          p.dK + ((row0 + k) * p.H + h) * D, key_ok, 0, D / 32);
        }
    }
    teardown<D>(tmem);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Before the one-pass kernel: D_i = dO_i . O_i for every (token, head) row of a
// dense [B, N, H, D] batch, stored [B, H, N] and, with lse_i log2 e, as pairs
// [B * H, n_pad] (zero pairs past N); and the dQ accumulator set to zero.
// D / 8 lanes take a row (16 bytes a lane; the same sum order as the dQ
// kernel's D); a warp keeps 8 rows' loads in flight.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *O,
                                                       const __nv_bfloat16 *dO, const float *lse,
                                                       float *Dv, float2 *stat2, float4 *acc,
                                                       int64_t acc_vec, int64_t rows, int H,
                                                       int N, int64_t n_pad)
{
    constexpr int kRowsPerWarp = 8;
    constexpr int kLanes = D / 8, kRowsPerInst = 32 / kLanes, kU = kRowsPerWarp / kRowsPerInst;
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < acc_vec; i += nthreads)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t bh_count = rows / N / H * H;
    const int64_t pads = bh_count * (n_pad - N);
    for (int64_t i = tid; i < pads; i += nthreads) {
        const int64_t bh = i / (n_pad - N), q = N + i % (n_pad - N);
        stat2[bh * n_pad + q] = make_float2(0.f, 0.f);
    }
    const int lane = threadIdx.x & 31, sub = lane / kLanes, l16 = lane % kLanes;
    for (int64_t base = (tid >> 5) * kRowsPerWarp; base < rows;
         base += (nthreads >> 5) * kRowsPerWarp) {
        // every load of the 8 rows first (the statistic's index and its lse
        // too, in the row's leading lane), then the dot products
        uint4 o[kU], g[kU];
        int64_t bhq[kU], sq[kU];
        float lv[kU];
        // (b, q, h) of the group's first row by division, the others by carry
        const int64_t token0 = base / H;
        const int h0 = int(base - token0 * H);
        const int64_t b0 = token0 / N, q0 = token0 - b0 * N;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t row = base + u * kRowsPerInst + sub;
            o[u] = make_uint4(0, 0, 0, 0);
            g[u] = o[u];
            lv[u] = 0.f;
            bhq[u] = sq[u] = 0;
            if (row < rows) {
                o[u] = reinterpret_cast<const uint4 *>(O + row * D)[l16];
                g[u] = reinterpret_cast<const uint4 *>(dO + row * D)[l16];
                if (l16 == 0) {
                    int hh = h0 + u * kRowsPerInst + sub;
                    int64_t q = q0, bb = b0;
                    while (hh >= H) {
                        hh -= H;
                        if (++q == N) {
                            q = 0;
                            ++bb;
                        }
                    }
                    const int64_t bh = bb * H + hh;
                    bhq[u] = bh * N + q;
                    sq[u] = bh * n_pad + q;
                    lv[u] = lse[bhq[u]];
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&o[u]);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&g[u]);
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = __bfloat1622float2(o2[e]), c = __bfloat1622float2(g2[e]);
                sum = fmaf(a.x, c.x, sum);
                sum = fmaf(a.y, c.y, sum);
            }
#pragma unroll
            for (int m = kLanes / 2; m > 0; m >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, m);
            if (l16 == 0 && base + u * kRowsPerInst + sub < rows) {
                Dv[bhq[u]] = sum;
                stat2[sq[u]] = make_float2(lv[u] * kLog2e, sum);
            }
        }
    }
}

// After it: dQ[b, q, h, :] = bf16(scale * acc[b H + h, q, :]), 8 elements per
// thread and iteration (two 16-byte loads, one 16-byte store), four iterations'
// loads in flight.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4 *acc, uint4 *dQ,
                                                             int64_t bh_count, int H, int N,
                                                             int64_t n_pad, float scale)
{
    constexpr int kVec = D / 8, kUnroll = 4;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the pass's sums are complete
    const int64_t n = bh_count * N * kVec;            // (b h, q < N, 8-element group)
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n;
         i0 += stride * kUnroll) {
        float4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t row = i / kVec, bh = row / N, q = row % N;
                const float4 *src = acc + (bh * n_pad + q) * (D / 4) + 2 * (i % kVec);
                a[u] = src[0];
                b[u] = src[1];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t row = i / kVec, bh = row / N, q = row % N;
                uint4 w;
                w.x = ptx::pack_bf16x2(scale * a[u].x, scale * a[u].y);
                w.y = ptx::pack_bf16x2(scale * a[u].z, scale * a[u].w);
                w.z = ptx::pack_bf16x2(scale * b[u].x, scale * b[u].y);
                w.w = ptx::pack_bf16x2(scale * b[u].z, scale * b[u].w);
                dQ[(((bh / H) * N + q) * H + bh % H) * kVec + i % kVec] = w;
            }
        }
    }
}

// The prep kernel for packed batches ([total, H, D] tensors, lse and D in
// [H, total]): D_i as above, the pairs in [H, B, n_pad] (sequence b's query q
// at (h B + b) n_pad + q, zero pairs past its length), the accumulator
// [H, total_pad, D] set to zero.  A row's sequence is found by binary search
// in cu_seqlens; rows outside every sequence, or past n_pad, write no pair.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_packed_kernel(
    const __nv_bfloat16 *O, const __nv_bfloat16 *dO, const float *lse, float *Dv, float2 *stat2,
    float4 *acc, int64_t acc_vec, const int32_t *cu_seqlens, int B, int H, int64_t total,
    int64_t n_pad)
{
    constexpr int kRowsPerWarp = 8;
    constexpr int kLanes = D / 8, kRowsPerInst = 32 / kLanes, kU = kRowsPerWarp / kRowsPerInst;
    const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = tid; i < acc_vec; i += nthreads)
        acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t n_pairs = int64_t(H) * B * n_pad;
    for (int64_t i = tid; i < n_pairs; i += nthreads) {
        const int b = int((i / n_pad) % B);
        const int64_t q = i % n_pad;
        if (q >= int64_t(cu_seqlens[b + 1]) - cu_seqlens[b])
            stat2[i] = make_float2(0.f, 0.f);
    }
    const int64_t rows = total * H;
    const int lane = threadIdx.x & 31, sub = lane / kLanes, l16 = lane % kLanes;
    for (int64_t base = (tid >> 5) * kRowsPerWarp; base < rows;
         base += (nthreads >> 5) * kRowsPerWarp) {
        // every load of the 8 rows first (the row's sequence, found by binary
        // search in cu_seqlens, and its lse too, in the row's leading lane),
        // then the dot products
        uint4 o[kU], g[kU];
        int64_t dq_[kU], sq[kU];
        float lv[kU];
        // (token, h) of the group's first row by division, the others by carry
        const int64_t token0 = base / H;
        const int h0 = int(base - token0 * H);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t row = base + u * kRowsPerInst + sub;
            o[u] = make_uint4(0, 0, 0, 0);
            g[u] = o[u];
            lv[u] = 0.f;
            dq_[u] = 0;
            sq[u] = -1;                              // no pair for this row
            if (row < rows) {
                o[u] = reinterpret_cast<const uint4 *>(O + row * D)[l16];
                g[u] = reinterpret_cast<const uint4 *>(dO + row * D)[l16];
                if (l16 == 0) {
                    int hh = h0 + u * kRowsPerInst + sub;
                    int64_t token = token0;
                    while (hh >= H) {
                        hh -= H;
                        ++token;
                    }
                    dq_[u] = int64_t(hh) * total + token;
                    lv[u] = lse[dq_[u]];
                    int lo = 0, hi = B;              // largest b with cu_seqlens[b] <= token
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (cu_seqlens[mid] <= token)
                            lo = mid;
                        else
                            hi = mid;
                    }
                    const int64_t q = token - cu_seqlens[lo];
                    if (q >= 0 && token < cu_seqlens[lo + 1] && q < n_pad)
                        sq[u] = (int64_t(hh) * B + lo) * n_pad + q;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const __nv_bfloat162 *o2 = reinterpret_cast<const __nv_bfloat162 *>(&o[u]);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&g[u]);
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a = __bfloat1622float2(o2[e]), c = __bfloat1622float2(g2[e]);
                sum = fmaf(a.x, c.x, sum);
                sum = fmaf(a.y, c.y, sum);
            }
#pragma unroll
            for (int m = kLanes / 2; m > 0; m >>= 1)
                sum += __shfl_xor_sync(0xffffffffu, sum, m);
            if (l16 == 0 && base + u * kRowsPerInst + sub < rows) {
                Dv[dq_[u]] = sum;
                if (sq[u] >= 0)
                    stat2[sq[u]] = make_float2(lv[u] * kLog2e, sum);
            }
        }
    }
}

// The conversion for packed batches: dQ[t, h, :] = bf16(scale *
// acc[h, t, :]) for t < total.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_convert_packed_kernel(const float4 *acc, uint4 *dQ,
                                                                    int H, int64_t total,
                                                                    int64_t total_pad, float scale)
{
    constexpr int kVec = D / 8, kUnroll = 4;
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the pass's sums are complete
    const int64_t n = int64_t(H) * total * kVec;      // (h, t, 8-element group)
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i0 < n;
         i0 += stride * kUnroll) {
        float4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t row = i / kVec, hh = row / total, t = row % total;
                const float4 *src = acc + (hh * total_pad + t) * (D / 4) + 2 * (i % kVec);
                a[u] = src[0];
                b[u] = src[1];
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n) {
                const int64_t row = i / kVec, hh = row / total, t = row % total;
                uint4 w;
                w.x = ptx::pack_bf16x2(scale * a[u].x, scale * a[u].y);
                w.y = ptx::pack_bf16x2(scale * a[u].z, scale * a[u].w);
                w.z = ptx::pack_bf16x2(scale * b[u].x, scale * b[u].y);
                w.w = ptx::pack_bf16x2(scale * b[u].z, scale * b[u].w);
                dQ[(t * H + hh) * kVec + i % kVec] = w;
            }
        }
    }
}

template <int D, bool PACKED>
int launch_bwd_d(const BwdParams &p_dq, const BwdParams &p_dkdv, cudaStream_t stream)
{
    auto kdq = attn_bwd_dq_kernel<D, PACKED>;
    auto kdkdv = attn_bwd_dkdv_kernel<D, PACKED>;
    static PerDeviceOnce once_dq, once_dkdv;
    if (!set_max_dynamic_smem(once_dq, reinterpret_cast<const void *>(kdq),
                              int(CfgQ<D>::kSmemBytes)) ||
        !set_max_dynamic_smem(once_dkdv, reinterpret_cast<const void *>(kdkdv),
                              int(Cfg<D>::kSmemBytes)))
        return FA_ERR_CUDA;
    const int64_t blocks = int64_t(p_dq.n_tiles) * p_dq.B * p_dq.H;
    kdq<<<dim3(unsigned(blocks)), dim3(kThreads), CfgQ<D>::kSmemBytes, stream>>>(p_dq);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    // the dK/dV kernel is a programmatic dependent of the dQ kernel (no early
    // trigger: it may start as the dQ kernel's CTAs exit; it waits for its
    // completion before reading D)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kdkdv, p_dkdv);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace {
// Groups of (sequence, head) pairs for a dense launch in which every tile CTA
// of a head streams `per_head` bytes of that head (the other side's tiles,
// and the dQ sums).  With all heads' heaviest tiles first, those bytes exceed
// L2 and are read again from DRAM; past half of L2 (64 MB) the heads run in
// consecutive groups of about 32 MB, as long as every group keeps at least
// 1.5 waves of CTAs.  1: one group.
int bwd_head_groups(int bh, int n_tiles, int64_t per_head, int sms)
{
    int best = 1;
    if (per_head * bh <= (int64_t(64) << 20) || sms <= 0)
        return best;
    for (int g = 2; g <= bh; ++g) {
        if (bh % g != 0)
            continue;
        if (2 * int64_t(n_tiles) * (bh / g) < 3 * int64_t(sms))
            break;
        best = g;
        if (per_head * (bh / g) <= (int64_t(32) << 20))
            break;
    }
    return best;
}

}  // namespace

int launch_attention_bwd(const AttnBwdArgs &a, cudaStream_t stream)
{
    BwdParams p;
    const int64_t total = a.cu_seqlens != nullptr ? a.total : int64_t(a.B) * a.N;
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
    p.n_sub = (a.N + BS - 1) / BS;
    p.scale = a.scale;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.err_word = a.err_word;
    p.cu_seqlens = a.cu_seqlens;
    p.total = total;
    p.expire_wait_ns = 0;
    const int64_t blocks = int64_t(p.n_tiles) * a.B * a.H;
    if (blocks == 0)
        return FA_OK;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    // the dQ kernel streams each head's K and V, the dK/dV kernel its Q and
    // dO: 4 N d bytes a head each
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FA_ERR_CUDA;
    p.head_groups = a.cu_seqlens != nullptr
                        ? 1
                        : bwd_head_groups(a.B * a.H, p.n_tiles, int64_t(4) * a.N * a.d, sms);
    BwdParams p_dq = p, p_dkdv = p;
    if (!make_tmap_bf16(&p_dq.tm_a0, a.Q, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dq.tm_a1, a.dO, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dq.tm_s0, a.K, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dq.tm_s1, a.V, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dkdv.tm_a0, a.K, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dkdv.tm_a1, a.V, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p_dkdv.tm_s0, a.Q, total, a.H, a.d, BS) ||
        !make_tmap_bf16(&p_dkdv.tm_s1, a.dO, total, a.H, a.d, BS))
        return FA_ERR_CUDA;
    // packed batches get their own instantiation, so that the dense kernels
    // keep the sequence length a kernel constant
    if (a.cu_seqlens != nullptr)
        return a.d == 64 ? launch_bwd_d<64, true>(p_dq, p_dkdv, stream)
                         : launch_bwd_d<128, true>(p_dq, p_dkdv, stream);
    return a.d == 64 ? launch_bwd_d<64, false>(p_dq, p_dkdv, stream)
                     : launch_bwd_d<128, false>(p_dq, p_dkdv, stream);
}

namespace {
// The one-pass form's three launches at head dim D.
template <int D>
int launch_bwd_atomic_d(const AttnBwdArgs &a, BwdParams &p, int64_t blocks, int64_t acc_floats,
                        int sms, cudaStream_t stream)
{
    const bool packed = a.cu_seqlens != nullptr;
    static PerDeviceOnce once_fused, once_fused_packed;
    auto kf = packed ? attn_bwd_fused_kernel<D, true> : attn_bwd_fused_kernel<D, false>;
    if (!set_max_dynamic_smem(packed ? once_fused_packed : once_fused,
                              reinterpret_cast<const void *>(kf), int(CfgF<D>::kSmemBytes)))
        return FA_ERR_CUDA;
    if (packed)
        bwd_prep_packed_kernel<D><<<dim3(unsigned(sms * 8)), dim3(256), 0, stream>>>(
            p.O, p.dO, a.lse, a.D, const_cast<float2 *>(p.stat2),
            reinterpret_cast<float4 *>(a.dq_acc), acc_floats / 4, a.cu_seqlens, a.B, a.H,
            p.total, p.n_pad);
    else
        bwd_prep_kernel<D><<<dim3(unsigned(sms * 8)), dim3(256), 0, stream>>>(
            p.O, p.dO, a.lse, a.D, const_cast<float2 *>(p.stat2),
            reinterpret_cast<float4 *>(a.dq_acc), acc_floats / 4, p.total * a.H, a.H, a.N,
            p.n_pad);
    if (cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    // the pass and the conversion are programmatic dependents of the kernel
    // before them (no early trigger: each may start as the previous one's
    // CTAs exit, and waits for its completion before reading its output)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = CfgF<D>::kSmemBytes;
    if (cudaLaunchKernelEx(&cfg, kf, p) != cudaSuccess || cudaGetLastError() != cudaSuccess)
        return FA_ERR_CUDA;
    cfg.gridDim = dim3(unsigned(sms * 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    const cudaError_t e =
        packed ? cudaLaunchKernelEx(&cfg, bwd_dq_convert_packed_kernel<D>,
                                    reinterpret_cast<const float4 *>(a.dq_acc),
                                    reinterpret_cast<uint4 *>(p.dQ), a.H, p.total, p.total_pad,
                                    a.scale)
               : cudaLaunchKernelEx(&cfg, bwd_dq_convert_kernel<D>,
                                    reinterpret_cast<const float4 *>(a.dq_acc),
                                    reinterpret_cast<uint4 *>(p.dQ), int64_t(a.B) * a.H, a.H,
                                    a.N, p.n_pad, a.scale);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
}  // namespace

int launch_attention_bwd_atomic(const AttnBwdArgs &a, cudaStream_t stream)
{
    if ((a.d != 64 && a.d != 128) || a.dq_acc == nullptr)
        return FA_ERR_UNSUPPORTED;
    const bool packed = a.cu_seqlens != nullptr;
    BwdParams p;
    const int64_t total = packed ? a.total : int64_t(a.B) * a.N;
    const int64_t n_pad = bwd_atomic_n_pad(a.N);
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
    p.n_sub = (a.N + BS - 1) / BS;
    p.scale = a.scale;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.err_word = a.err_word;
    p.cu_seqlens = a.cu_seqlens;
    p.total = total;
    p.dq_acc = a.dq_acc;
    p.n_pad = n_pad;
    p.total_pad = total + 64;
    // workspace: the accumulator, then the (lse log2 e, D) pairs
    const int64_t acc_floats = packed ? int64_t(a.H) * p.total_pad * a.d
                                      : int64_t(a.B) * a.H * n_pad * a.d;
    p.stat2 = reinterpret_cast<const float2 *>(a.dq_acc + acc_floats);
    const int64_t blocks = int64_t(p.n_tiles) * a.B * a.H;
    if (blocks == 0 || total == 0)
        return FA_OK;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    if (!make_tmap_bf16(&p.tm_a0, a.K, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p.tm_a1, a.V, total, a.H, a.d, BT) ||
        !make_tmap_bf16(&p.tm_s0, a.Q, total, a.H, a.d, BS) ||
        !make_tmap_bf16(&p.tm_s1, a.dO, total, a.H, a.d, BS))
        return FA_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FA_ERR_CUDA;
    // every key-tile CTA of a head streams the head's Q and dO and adds into
    // its dQ sums: 8 N d bytes a head
    p.head_groups = packed ? 1 : bwd_head_groups(a.B * a.H, p.n_tiles, int64_t(8) * a.N * a.d, sms);
    p.expire_wait_ns = a.expire_wait_ns;
    return a.d == 64 ? launch_bwd_atomic_d<64>(a, p, blocks, acc_floats, sms, stream)
                     : launch_bwd_atomic_d<128>(a, p, blocks, acc_floats, sms, stream);
}

}  // namespace fa
