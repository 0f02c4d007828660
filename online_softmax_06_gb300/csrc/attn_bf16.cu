// attn_bf16.cu -- exact attention forward on the sm_103a tensor cores.
//
// What it computes: O = softmax(scale * Q K^T + mask) V and the row logsumexp,
// tile by tile with the online-softmax recurrence of "第二十二课：Softmax 为什么难以
// 高效…" (lincklin.cn) §三十二 and "少搬一趟：FlashAttention 四代进化史" §2.2: for each
// K/V tile the running row max m, running sum l and the unnormalised output o~
// are updated (o~ and l rescaled by exp(m_old - m_new)), and O = o~ / l and
// lse = m + ln l are written once at the end (§3.2 deferred normalisation,
// §2.4 logsumexp).  S and P never leave the chip.
//
// How it maps to a GB300 SM (the booklet's §5.5 pipeline for Blackwell is the
// starting point; everything here is written for tcgen05 from the PTX ISA):
//   * one CTA per SM, 320 threads, owns two 128-row Q tiles of one
//     (sequence, head) -- "Q0" and "Q1", adjacent in the sequence -- so every
//     K/V tile loaded into shared memory feeds 2 x 128 rows;
//   * warp 8 (one lane) issues TMA loads: Q0, K_0, Q1 (one barrier per Q tile,
//     so the first Q0 K_0^T does not wait for Q1), then V_0, K_1, V_1, ...
//     into a ring of shared-memory stages guarded by full/empty mbarriers;
//   * warp 9 owns the tensor memory and issues every tcgen05.mma (the whole
//     warp runs the issuing loop and its barrier waits converged, and one
//     elected lane issues: the loop's descriptors stay warp-uniform, which
//     keeps the issue rate at the tensor pipe's rate):
//     S_t = Q_t K_j^T (bf16 x bf16 -> fp32, M=N=128, K=d) into TMEM, and
//     O_t += P_t V_j with P_t read from TMEM (written there by the softmax
//     threads over the upper half of S_t) and V_j from shared memory as an
//     MN-major operand; the issue order QK0, QK1, PV0, QK0', PV1, QK1', ...
//     lets one tile's softmax run while the other tile's MMAs execute;
//   * warps 0-3 and 4-7 are the softmax warpgroups of Q0 and Q1: thread r owns
//     query row r (TMEM lane r), loads its 128 scores with tcgen05.ld, applies
//     the causal / sequence-end mask on the tiles that need it, updates m and
//     l, converts P to bf16 into TMEM, and rescales its row of O in TMEM only
//     when its maximum grew (warp-uniform skip otherwise); after the last tile
//     it normalises O and writes lse (fp32) and O (bf16): a whole tile is
//     written into the Q tile's shared-memory buffer (free by then, and laid
//     out as the TMA box) and leaves in one TMA store; a tile that runs past
//     the end of its sequence is stored row by row.
// Tensor memory per CTA (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d),
// O1 [256+d, 256+2d); P_t aliases columns 64..127 of S_t.
// Every wait is bounded (ptx::mbar_wait); a timed-out wait raises an error bit,
// all roles leave their loops, in-flight copies and MMAs are drained, and the
// CTA frees its tensor memory and exits.
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

constexpr int BM = 128;              // query rows per Q tile
constexpr int BN = 128;              // keys per K/V tile
constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColPinS = 64;    // P_t starts 64 columns into S_t
constexpr float kLn2 = 0.69314718055994531f;
constexpr float kRescaleLog2 = 8.f;  // move the reference max only past 2^8

// TMEM column of S_t and of O_t (t = 0, 1) for head dimension D.
__device__ __forceinline__ uint32_t col_s(int t) { return uint32_t(t) * 128u; }
template <int D>
__device__ __forceinline__ uint32_t col_o(int t) { return 256u + uint32_t(t) * D; }
constexpr uint32_t kChunkBytes = BM * 128;  // 128 rows x 128 bytes (64 bf16)

// FP8: Q, K and V arrive as e4m3 (one byte per element; V transposed per
// head, keys contiguous), so a 128-row tile of d = 128 is one 128-byte chunk.
template <int D, bool FP8 = false>
struct Cfg {
    static constexpr int kChunks = FP8 ? 1 : D / 64;        // 128-byte column chunks
    static constexpr uint32_t kTileBytes = BM * D * (FP8 ? 1 : 2);   // one Q, K or V tile
    static constexpr int kStages = (D == 128 && !FP8) ? 4 : 8;      // K/V ring depth
    // a Q buffer also stages the tile's bf16 O for the epilogue's TMA store
    static constexpr uint32_t kQBytes = BM * D * 2;
    // shared memory: [Q0][Q1][ring x kStages][barriers, flags]
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffRing = 2 * kQBytes;
    static constexpr uint32_t kOffBar = kOffRing + kStages * kTileBytes;
    static constexpr uint32_t kBarBytes = 8 * (2 + 2 * kStages + 2 + 2 + 2 + 1 + 1);
    static constexpr uint32_t kSmemBytes = kOffBar + kBarBytes + 16 + 1024;  // +1024 align slack
};

struct Bf16Params {
    CUtensorMap tm_q, tm_k, tm_v;    // 3-D maps over [rows, H, d] bf16, box {64, 1, 128}
    CUtensorMap tm_o;                // the same over O (stores of whole tiles)
    // FP8: tm_q, tm_k are e4m3 row maps, tm_v the transposed V' map; the
    // scores are (Q'K'^T) sq[tile] sk[tile] and O = (P V') sv
    const float *sq, *sk, *sv;       // [B, H, n_tiles], [B, H, n_tiles], [B, H]
    int n_tiles;
    __nv_bfloat16 *O;
    float *lse;
    int B, H, N;                     // N: queries per sequence (dense) / longest sequence
    int H_row;                       // heads per token row of Q/K/V/O and per (b) in lse
    int Nk;                          // keys per sequence (dense); packed batches use L
    int n_pairs;                     // Q-tile pairs per (sequence, head) at length N
    int head_groups;                 // the (sequence, head) pairs in this many consecutive
                                     // groups, heaviest Q-tile pairs first within each
    int64_t total;                   // query rows of Q / O
    float scale_log2;                // scale * log2(e)
    int causal;
    int kv_off;                      // causal: query i sees keys j <= i + kv_off
    int splits;                      // key ranges per Q-tile pair (1: write O, lse)
    float *O_accum;                  // splits > 1: [splits, B, N, H, d] fp32 partial O
    float *lse_accum;                // splits > 1: [splits, B, H, N] fp32 partial lse
    const int32_t *cu_seqlens;
    // split-KV on packed batches: key rows per sequence (cu_seqlens then
    // holds the query rows); causal is bottom-right within each sequence
    const int32_t *cu_seqlens_k;
    int64_t total_k;                 // rows of K / V
    int *err_word;
    uint32_t expire_wait_ns;         // failure-detection test only (0: off)
};

struct Barriers {
    uint64_t *q_full, *kv_full, *kv_empty, *s_full, *p_full, *o_full, *drain;
    uint64_t *never;                 // nothing arrives: the failure-detection test waits here
};

// Bounded wait used only while draining after an abort: ignores the abort flag.
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

// SPLIT: compiled for split-KV calls (key ranges, query/key lengths that
// differ, partial outputs); the plain instantiation has one range per pair and
// kv_off = 0, so that logic folds away.
template <int D, bool SPLIT, bool FP8 = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ Bf16Params p)
{
    static_assert(!FP8 || (D == 128 && !SPLIT), "FP8: d = 128, no key splits");
    // FP8: launched as a programmatic dependent of the V transpose; nothing
    // the quantisation wrote is read before this wait returns
    if constexpr (FP8)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    using C = Cfg<D, FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    Barriers bar;
    bar.q_full = bars;                         // one per Q tile
    bar.kv_full = bars + 2;
    bar.kv_empty = bars + 2 + C::kStages;
    bar.s_full = bars + 2 + 2 * C::kStages;
    bar.p_full = bar.s_full + 2;
    bar.o_full = bar.p_full + 2;
    bar.drain = bar.o_full + 2;
    bar.never = bar.drain + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + (C::kBarBytes / 8));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    // ---- work item: (sequence b, head h, Q-tile pair, key split), heaviest
    //      pairs first within each group of (sequence, head) pairs (the
    //      groups run one after another, so only a group's K/V compete for
    //      L2) ----------------------------------------------------------------------
    const int bh_count = p.B * p.H;
    const int n_splits = SPLIT ? p.splits : 1;
    int kv_off = SPLIT ? p.kv_off : 0;
    const int split = SPLIT ? int(blockIdx.x % unsigned(n_splits)) : 0;
    const int rest = SPLIT ? int(blockIdx.x / unsigned(n_splits)) : int(blockIdx.x);
    int pair, bh;
    if (SPLIT || FP8 || p.head_groups <= 1) {   // (FP8: K', V' are small enough for L2)
        pair = p.n_pairs - 1 - rest / bh_count;
        bh = rest % bh_count;
    } else {
        const int gsz = bh_count / p.head_groups;           // pairs per group
        const int grp = rest / (p.n_pairs * gsz);
        const int in_grp = rest - grp * (p.n_pairs * gsz);
        pair = p.n_pairs - 1 - in_grp / gsz;
        bh = grp * gsz + in_grp % gsz;
    }
    const int b = bh / p.H, h = bh % p.H;
    int64_t start, start_k;    // first query row / first key row of the sequence
    int L, Lk;                 // query and key counts of the sequence
    if (p.cu_seqlens != nullptr) {
        const int64_t s0 = p.cu_seqlens[b], s1 = p.cu_seqlens[b + 1];
        if (s0 < 0 || s1 < s0 || s1 > p.total || s1 - s0 > p.N) {
            if (threadIdx.x == 0 && pair == 0 && h == 0 && split == 0)
                record_device_error(p.err_word, FA_DEVERR_BAD_SEQLENS);
            return;
        }
        start = start_k = s0;
        L = Lk = int(s1 - s0);
        if (SPLIT && p.cu_seqlens_k != nullptr) {
            const int64_t k0 = p.cu_seqlens_k[b], k1 = p.cu_seqlens_k[b + 1];
            if (k0 < 0 || k1 < k0 || k1 > p.total_k || k1 - k0 > p.Nk ||
                (p.causal && k1 - k0 < L)) {
                if (threadIdx.x == 0 && pair == 0 && h == 0 && split == 0)
                    record_device_error(p.err_word, FA_DEVERR_BAD_SEQLENS);
                return;
            }
            start_k = k0;
            Lk = int(k1 - k0);
            kv_off = Lk - L;
        }
    } else {
        start = int64_t(b) * p.N;
        L = p.N;
        start_k = SPLIT ? int64_t(b) * p.Nk : start;
        Lk = SPLIT ? p.Nk : L;
    }
    const int qt0 = 2 * pair;                  // Q0 = tile qt0, Q1 = tile qt0 + 1
    if (qt0 * BM >= L)
        return;                                // whole CTA: nothing to do
    // Split-KV partial results: [splits, B, N, H, d] and [splits, B, H, N]
    // dense; packed batches use [splits, total, H, d] and [splits, H, total]
    const bool packed = p.cu_seqlens != nullptr;
    auto lse_acc_index = [&](int i) -> int64_t {
        return packed ? (int64_t(split) * p.H + h) * p.total + start + i
                      : ((int64_t(split) * p.B + b) * p.H + h) * p.N + i;
    };
    const bool has_q1 = (qt0 + 1) * BM < L;
    const int n_kv = (Lk + BN - 1) / BN;
    int n0, n1, n_max, j0 = 0;
    if constexpr (SPLIT) {
        // K/V tiles a Q tile sees: when causal, up to the one holding key
        // (last row of the tile) + kv_off
        auto tiles_seen = [&](int qt) {
            if (!p.causal)
                return n_kv;
            const int last = (qt * BM + BM - 1 + kv_off) / BN + 1;
            return last < n_kv ? last : n_kv;
        };
        const int n0_all = tiles_seen(qt0);
        const int n1_all = has_q1 ? tiles_seen(qt0 + 1) : 0;
        const int n_all = n0_all > n1_all ? n0_all : n1_all;
        // this split's key tiles [j0, j0 + chunk) of the pair's range; a tile
        // takes the steps of that range its keys reach (possibly none)
        const int chunk = (n_all + n_splits - 1) / n_splits;
        j0 = split * chunk;
        auto steps = [&](int n_t) {
            const int e = n_t < j0 + chunk ? n_t : j0 + chunk;
            return e > j0 ? e - j0 : 0;
        };
        n0 = steps(n0_all);
        n1 = steps(n1_all);
    } else {
        n0 = p.causal ? qt0 + 1 : n_kv;
        n1 = has_q1 ? (p.causal ? qt0 + 2 : n_kv) : 0;
    }
    n_max = n0 > n1 ? n0 : n1;
    if (SPLIT && n_max == 0) {
        // an empty split: its partial result for the pair's rows is empty
        // (lse = -inf, weight 0 in the combine).  With one split this happens
        // only for a packed sequence without keys: its rows see no key, so O
        // is 0 and lse is -inf.
        if (threadIdx.x < 2 * BM) {
            const int i = qt0 * BM + int(threadIdx.x);
            if (i < L && n_splits > 1) {
                p.lse_accum[lse_acc_index(i)] = -INFINITY;
            } else if (i < L) {
                uint4 *orow = reinterpret_cast<uint4 *>(p.O + ((start + i) * p.H_row + h) * D);
#pragma unroll
                for (int q = 0; q < D / 8; ++q)
                    orow[q] = make_uint4(0, 0, 0, 0);
                if (packed)
                    p.lse[int64_t(h) * p.total + start + i] = -INFINITY;
                else
                    p.lse[(int64_t(b) * p.H_row + h) * p.N + i] = -INFINITY;
            }
        }
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- set-up: barriers, tensor memory ----------------------------------
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar.q_full[0], 1);
        ptx::mbar_init(&bar.q_full[1], 1);
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(&bar.kv_full[s], 1);
            ptx::mbar_init(&bar.kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(&bar.s_full[t], 1);
            ptx::mbar_init(&bar.p_full[t], 128);
            ptx::mbar_init(&bar.o_full[t], 1);
        }
        ptx::mbar_init(bar.drain, 1);
        ptx::mbar_init(bar.never, 1);
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
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    bool aborted = false;

    uint8_t *q_smem[2] = {smem + C::kOffQ, smem + C::kOffQ + C::kQBytes};
    uint8_t *ring = smem + C::kOffRing;

    if (warp == kWarpLoad) {
        // ======================= TMA producer ==============================
        if (lane == 0) {
            int last_phase[C::kStages];
            for (int s = 0; s < C::kStages; ++s)
                last_phase[s] = -1;
            // Q0 (if it has key tiles here), then K_0, then Q1: the first
            // Q0 K_0^T can start before Q1 has landed
            bool q_issued[2] = {false, false};
            auto load_q = [&](int t) {
                q_issued[t] = true;
                ptx::mbar_arrive_expect_tx(&bar.q_full[t], C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    ptx::tma_load_3d(q_smem[t] + c * kChunkBytes, &p.tm_q, &bar.q_full[t], c * 64, h,
                                     int(start + int64_t(qt0 + t) * BM));
            };
            if (n0 > 0)
                load_q(0);
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < n_max && !aborted; ++j) {
                for (int kv = 0; kv < 2; ++kv) {
                    if (!ptx::mbar_wait(&bar.kv_empty[stage], phase ^ 1u, abort_flag,
                                        p.err_word)) {
                        aborted = true;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&bar.kv_full[stage], C::kTileBytes);
                    const CUtensorMap *tm = kv ? &p.tm_v : &p.tm_k;
                    if (FP8 && kv) {
                        // V'^T rows (b, h, 0 .. d-1), keys of this tile
                        ptx::tma_load_2d(ring + stage * C::kTileBytes, tm, &bar.kv_full[stage],
                                         (j0 + j) * BN, (b * p.H + h) * D);
                    } else {
                        for (int c = 0; c < C::kChunks; ++c)
                            ptx::tma_load_3d(ring + stage * C::kTileBytes + c * kChunkBytes, tm,
                                             &bar.kv_full[stage], c * 64, h,
                                             int(start_k + int64_t(j0 + j) * BN));
                    }
                    last_phase[stage] = int(phase);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (j == 0 && kv == 0 && n1 > 0)
                        load_q(1);
                }
            }
            if (aborted || *abort_flag) {
                // let every copy already issued land before the CTA goes away
                for (int t = 0; t < 2; ++t)
                    if (q_issued[t])
                        drain_wait(&bar.q_full[t], 0);
                for (int s = 0; s < C::kStages; ++s)
                    if (last_phase[s] >= 0)
                        drain_wait(&bar.kv_full[s], uint32_t(last_phase[s]));
            }
        }
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ======================= MMA issuer (whole warp) =====================
        {
            constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, true);
            constexpr uint64_t desc_kmajor = ptx::smem_desc_base(16, 1024);
            constexpr uint64_t desc_mnmajor = ptx::smem_desc_base(kChunkBytes, 1024);
            // A descriptor built for a tile's base address is advanced to a
            // sub-block by adding (byte offset >> 4) to it: the start-address
            // field sits in the low 14 bits and every shared-memory address
            // here is below 256 KB, so the add never carries out of the field.
            const uint64_t dq0 = ptx::smem_desc(desc_kmajor, ptx::smem_u32(q_smem[0]));
            const uint64_t dq1 = ptx::smem_desc(desc_kmajor, ptx::smem_u32(q_smem[1]));
            const uint32_t ring_addr = ptx::smem_u32(ring);

            auto issue_qk = [&](int t, uint64_t dk) {
                const uint64_t dq = t == 0 ? dq0 : dq1;
                const uint32_t ts = tmem + col_s(t);
                if (ptx::elect_one()) {
                if constexpr (FP8) {
                    // e4m3: K = 32 per MMA, 32 bytes along the 128-byte row
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk)
                        ptx::mma_ss_f8(ts, dq + ((kk * 32) >> 4), dk + ((kk * 32) >> 4),
                                       ptx::idesc_e4m3_f32(BM, BN), kk > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
                        ptx::mma_ss(ts, dq + off, dk + off, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                }
                ptx::mma_commit(&bar.s_full[t]);
                }
                __syncwarp();
            };
            auto issue_pv = [&](int t, uint64_t dv, bool accumulate) {
                const uint32_t to = tmem + col_o<D>(t);
                const uint32_t tp = tmem + col_s(t) + kColPinS;
                if (ptx::elect_one()) {
                if constexpr (FP8) {
                    // P' e4m3 in TMEM (4 per column), V'^T K-major (keys contiguous)
#pragma unroll
                    for (int kk = 0; kk < BN / 32; ++kk)
                        ptx::mma_ts_f8(to, tp + kk * 8, dv + uint64_t((kk * 32) >> 4),
                                       ptx::idesc_e4m3_f32(BM, D), (accumulate || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        ptx::mma_ts(to, tp + kk * 8, dv + uint64_t((kk * 16 * 128) >> 4), idesc_pv,
                                    (accumulate || kk > 0) ? 1u : 0u);
                }
                }
                __syncwarp();
            };
            auto commit = [&](uint64_t *bar_) {
                if (ptx::elect_one())
                    ptx::mma_commit(bar_);
                __syncwarp();
            };

            int stage = 0;
            uint32_t phase = 0;
            // waits for the next ring stage; returns its K-major and MN-major
            // descriptors (the stage holds a K tile or a V tile)
            auto next_stage = [&](uint64_t &dk, uint64_t &dv) -> bool {
                if (!ptx::mbar_wait_warp(&bar.kv_full[stage], phase, abort_flag, p.err_word))
                    return false;
                const uint32_t addr = ring_addr + stage * C::kTileBytes;
                dk = ptx::smem_desc(desc_kmajor, addr);
                dv = ptx::smem_desc(FP8 ? desc_kmajor : desc_mnmajor, addr);
                return true;
            };
            auto advance = [&]() {
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };

            // Failure-detection test: a wait on a barrier that nothing arrives
            // at runs out after expire_wait_ns; it raises the error bit and the
            // abort flag, and the CTA winds down as after any timed-out wait.
            if (p.expire_wait_ns != 0u &&
                !__all_sync(0xffffffffu, ptx::mbar_wait_limited(bar.never, 0, abort_flag,
                                                                p.err_word, p.expire_wait_ns)))
                aborted = true;

            if (aborted) {
                // nothing issued: go straight to the drain below
            } else do {
                uint64_t k_desc, unused;
                if (!next_stage(k_desc, unused)) {
                    aborted = true;
                    break;
                }
                int k_stage = stage;
                advance();
                bool q_ok = true;
                for (int t = 0; t < 2 && q_ok; ++t) {
                    if ((t == 0 ? n0 : n1) == 0)
                        continue;
                    q_ok = ptx::mbar_wait_warp(&bar.q_full[t], 0, abort_flag, p.err_word);
                    if (q_ok) {
                        ptx::tc_fence_after_sync();
                        issue_qk(t, k_desc);
                    }
                }
                if (!q_ok) {
                    aborted = true;
                    break;
                }
                commit(&bar.kv_empty[k_stage]);

                for (int j = 0; j < n_max; ++j) {
                    uint64_t v_desc;
                    if (!next_stage(unused, v_desc)) {
                        aborted = true;
                        break;
                    }
                    const int v_stage = stage;
                    advance();
                    if (j < n0) {
                        if (!ptx::mbar_wait_warp(&bar.p_full[0], uint32_t(j) & 1u, abort_flag,
                                            p.err_word)) {
                            aborted = true;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        issue_pv(0, v_desc, j > 0);
                        if (j == n0 - 1)
                            commit(&bar.o_full[0]);
                    }
                    const bool more = j + 1 < n_max;
                    if (more) {
                        if (!next_stage(k_desc, unused)) {
                            aborted = true;
                            break;
                        }
                        k_stage = stage;
                        advance();
                        ptx::tc_fence_after_sync();
                        if (j + 1 < n0)
                            issue_qk(0, k_desc);
                    }
                    if (j < n1) {
                        if (!ptx::mbar_wait_warp(&bar.p_full[1], uint32_t(j) & 1u, abort_flag,
                                            p.err_word)) {
                            aborted = true;
                            break;
                        }
                        ptx::tc_fence_after_sync();
                        issue_pv(1, v_desc, j > 0);
                        if (j == n1 - 1)
                            commit(&bar.o_full[1]);
                    }
                    commit(&bar.kv_empty[v_stage]);
                    if (more) {
                        if (j + 1 < n1)
                            issue_qk(1, k_desc);
                        commit(&bar.kv_empty[k_stage]);
                    }
                }
            } while (false);
            // Every MMA issued above has completed (and every commit has arrived)
            // once this last commit arrives.
            if (ptx::elect_one()) {
                ptx::mma_commit(bar.drain);
                drain_wait(bar.drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ======================= softmax warpgroups ========================
        const int t = warp >> 2;                       // 0: Q0, 1: Q1
        const int r = threadIdx.x & 127;               // row in the Q tile = TMEM lane
        const int n_t = t == 0 ? n0 : n1;
        const int qt = qt0 + t;
        const int i = qt * BM + r;                     // query position in the sequence
        const uint32_t lane_bits = uint32_t((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_bits + col_s(t);
        const uint32_t tO = tmem + lane_bits + col_o<D>(t);
        float sl = p.scale_log2;
        if constexpr (FP8)                             // dequantise Q' K'^T: x sq sk
            sl *= p.sq[(int64_t(b) * p.H + h) * p.n_tiles + qt];
        float m = -INFINITY;                           // reference max, log2 units
        float l = 0.f;                                 // running sum (lse)
        // The running sum that divides O: l plus, per tile, the bf16 rounding
        // error of the tile's largest probability.  Under the conditional
        // rescale that probability is 2^(tile max - m), up to 2^8, not 1, and
        // its rounding (up to 2^-8 relative) enters P V; adding it here keeps
        // O a weighted mean of V rows for a row dominated by one key.
        float l_o = 0.f;

        for (int j = 0; j < n_t; ++j) {
            if (!ptx::mbar_wait(&bar.s_full[t], uint32_t(j) & 1u, abort_flag, p.err_word)) {
                aborted = true;
                break;
            }
            ptx::tc_fence_after_sync();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                ptx::tmem_ld32(tS + c * 32, sr[c]);
            ptx::tmem_wait_ld();

            // mask: keys past the causal bound (query i sees keys <= i + kv_off)
            // and past the end of the sequence's keys; jg is the key tile
            const int jg = j0 + j;
            bool diag, tail;
            int lim_causal, lim_len;
            if constexpr (SPLIT) {
                diag = p.causal && jg * BN + BN - 1 > qt * BM + kv_off;
                tail = (jg + 1) * BN > Lk;
                lim_causal = diag ? i + kv_off - jg * BN : BN - 1;  // last visible column
                lim_len = Lk - 1 - jg * BN;
            } else {
                diag = p.causal && j == qt;   // the diagonal tile (one range, kv_off = 0)
                tail = (j + 1) * BN > L;
                lim_causal = diag ? i - j * BN : BN - 1;
                lim_len = L - 1 - j * BN;
            }
            if (diag || tail) {
                const int lim = lim_causal < lim_len ? lim_causal : lim_len;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (c * 32 + e > lim)
                            sr[c][e] = __float_as_uint(-INFINITY);
            }
            // row maximum: three-input maxes over four independent chains
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int q = 0; q < 16; ++q)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = q * 8 + 2 * k;
                    m4[k] = ptx::max3(m4[k], __uint_as_float(sr[c >> 5][c & 31]),
                                      __uint_as_float(sr[(c + 1) >> 5][(c + 1) & 31]));
                }
            const float mx = fmaxf(ptx::max3(m4[0], m4[1], m4[2]), m4[3]);
            // Conditional rescale (booklet §5.4): the row keeps a reference
            // maximum m and moves it only when the tile maximum exceeds it by
            // more than kRescaleLog2, so every p stays <= 2^kRescaleLog2 (far
            // from overflow) while o~ is rescaled only on rare tiles.  o~ and l
            // share the reference, so it cancels in o~ / l and in
            // lse = m + log2 l: the result is exact for any reference.
            float slj = sl;
            if constexpr (FP8)
                slj *= p.sk[(int64_t(b) * p.H + h) * p.n_tiles + (j0 + j)];
            const float mt = mx * slj;
            const bool grew = mt > m + kRescaleLog2;
            const float m_new = grew ? mt : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = grew ? ptx::ex2(m - m_use) : 1.f;   // 0 on the first tile

            // P = exp2(s * sl - m) in bf16 into P_t's columns; the exponent
            // arguments are formed two at a time (packed fp32x2 FMA).
            const uint32_t tP = tS + kColPinS;
            const float2 sl2 = make_float2(slj, slj);
            const float2 nm2 = make_float2(-m_use, -m_use);
            // the row sum is accumulated two lanes at a time (packed fp32x2 add)
            float2 rowsum2 = make_float2(0.f, 0.f);
            if constexpr (FP8) {
                // P' = e4m3(p) four per column over columns 64..95 of S_t (p <=
                // 2^kRescaleLog2 < 448, so nothing saturates)
                uint32_t pk[32];
#pragma unroll
                for (int q4 = 0; q4 < 32; ++q4) {
                    const int col = 4 * q4;
                    const float2 a = __ffma2_rn(
                        make_float2(__uint_as_float(sr[col >> 5][col & 31]),
                                    __uint_as_float(sr[col >> 5][(col + 1) & 31])),
                        sl2, nm2);
                    const float2 c = __ffma2_rn(
                        make_float2(__uint_as_float(sr[col >> 5][(col + 2) & 31]),
                                    __uint_as_float(sr[col >> 5][(col + 3) & 31])),
                        sl2, nm2);
                    const float p0 = ptx::ex2(a.x), p1 = ptx::ex2(a.y);
                    const float p2 = ptx::ex2(c.x), p3 = ptx::ex2(c.y);
                    rowsum2 = __fadd2_rn(rowsum2, __fadd2_rn(make_float2(p0, p1),
                                                             make_float2(p2, p3)));
                    pk[q4] = ptx::pack_e4m3x4(p0, p1, p2, p3);
                }
                ptx::tmem_st32(tP, pk);
            } else
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = half * 64 + 2 * e;
                    const float2 sv = make_float2(__uint_as_float(sr[col >> 5][col & 31]),
                                                  __uint_as_float(sr[(col + 1) >> 5][(col + 1) & 31]));
                    const float2 arg = __ffma2_rn(sv, sl2, nm2);
                    const float p0 = ptx::ex2(arg.x), p1 = ptx::ex2(arg.y);
                    rowsum2 = __fadd2_rn(rowsum2, make_float2(p0, p1));
                    pk[e] = ptx::pack_bf16x2(p0, p1);
                }
                ptx::tmem_st32(tP + half * 32, pk);
            }
            // rescale this row of O~ when its reference moved (never on the
            // first tile: the first P V overwrites O); the warp goes together,
            // lanes whose reference did not move multiply by exactly 1
            if (j > 0 && __any_sync(0xffffffffu, grew)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + c * 32, o);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
                    ptx::tmem_st32(tO + c * 32, o);
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            ptx::mbar_arrive(&bar.p_full[t]);

            // The row sums are needed only after the last tile: they are
            // updated after P is handed over, off the path to the next MMA.
            const float tile_sum = rowsum2.x + rowsum2.y;
            l = l * corr + tile_sum;
            if constexpr (FP8) {
                l_o = l;
            } else {
                // the tile maximum's probability exactly as the loop formed
                // it (same fma and ex2), and its bf16 value
                const float p_top = ptx::ex2(fmaf(mx, slj, -m_use));
                const float p_top_bf16 = __uint_as_float(ptx::pack_bf16x2(p_top, 0.f) << 16);
                l_o = l_o * corr + (tile_sum + (p_top_bf16 - p_top));
            }
            m = m_new;
        }

        // ---- epilogue: O = O~ / l (bf16), lse = (m + log2 l) * ln 2 -----------
        // With several key splits the partial O (fp32) and lse of this split are
        // written instead; a row that saw no key in this split (possible only
        // there) gets lse = -inf, which gives it weight 0 in the combine.
        if constexpr (SPLIT) {
            if (!aborted && n_t > 0) {
                if (ptx::mbar_wait(&bar.o_full[t], 0, abort_flag, p.err_word)) {
                    ptx::tc_fence_after_sync();
                    const bool row_ok = i < L;
                    const bool empty = !(l > 0.f);
                    const float inv = empty ? 0.f : 1.f / l_o;
                    __nv_bfloat16 *orow = p.O + ((start + i) * p.H_row + h) * D;
                    const int64_t acc_rows = packed ? p.total : int64_t(p.B) * p.N;
                    const int64_t acc_row0 = packed ? start : int64_t(b) * p.N;
                    float *arow = p.O_accum +
                                  ((int64_t(split) * acc_rows + acc_row0 + i) * p.H + h) * D;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        ptx::tmem_ld32(tO + c * 32, o);
                        ptx::tmem_wait_ld();
                        if (!row_ok)
                            continue;
                        if (n_splits > 1) {
                            float4 *dst = reinterpret_cast<float4 *>(arow + c * 32);
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                dst[q] = make_float4(__uint_as_float(o[4 * q + 0]) * inv,
                                                     __uint_as_float(o[4 * q + 1]) * inv,
                                                     __uint_as_float(o[4 * q + 2]) * inv,
                                                     __uint_as_float(o[4 * q + 3]) * inv);
                            continue;
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 w;
                            w.x = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv,
                                                   __uint_as_float(o[8 * q + 1]) * inv);
                            w.y = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv,
                                                   __uint_as_float(o[8 * q + 3]) * inv);
                            w.z = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv,
                                                   __uint_as_float(o[8 * q + 5]) * inv);
                            w.w = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv,
                                                   __uint_as_float(o[8 * q + 7]) * inv);
                            dst[q] = w;
                        }
                    }
                    if (row_ok) {
                        const float lse = empty ? -INFINITY : (m + log2f(l)) * kLn2;
                        if (n_splits > 1)
                            p.lse_accum[lse_acc_index(i)] = lse;
                        else if (packed)
                            p.lse[int64_t(h) * p.total + start + i] = lse;
                        else
                            p.lse[(int64_t(b) * p.H_row + h) * p.N + i] = lse;
                    }
                }
            } else if (!aborted && n_splits > 1 && i < L) {
                // this tile has no keys in this split
                p.lse_accum[lse_acc_index(i)] = -INFINITY;
            }
        } else if (n_t > 0) {
            // A whole tile goes out through shared memory and one TMA store:
            // Q_t's buffer is free (every Q_t K^T completed before the last S_t
            // was published) and has the store's swizzled layout.  A tile that
            // runs past the end of its sequence is stored row by row, so that
            // no row of the next sequence is touched.
            const bool full_tile = (qt + 1) * BM <= L;
            uint8_t *o_stage = q_smem[t];
            const bool ok = !aborted && ptx::mbar_wait(&bar.o_full[t], 0, abort_flag, p.err_word);
            if (ok) {
                ptx::tc_fence_after_sync();
                const float inv = (FP8 ? p.sv[int64_t(b) * p.H + h] : 1.f) / l_o;
                const bool row_ok = i < L;
                __nv_bfloat16 *orow = p.O + ((start + i) * p.H_row + h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    ptx::tmem_ld32(tO + c * 32, o);
                    ptx::tmem_wait_ld();
                    uint4 w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        w[q].x = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv,
                                                  __uint_as_float(o[8 * q + 1]) * inv);
                        w[q].y = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv,
                                                  __uint_as_float(o[8 * q + 3]) * inv);
                        w[q].z = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv,
                                                  __uint_as_float(o[8 * q + 5]) * inv);
                        w[q].w = ptx::pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv,
                                                  __uint_as_float(o[8 * q + 7]) * inv);
                    }
                    if (full_tile) {
                        // 128-byte swizzle: 16-byte unit u of row r sits at
                        // unit position u ^ (r % 8) of the row's 128 bytes
                        uint8_t *rowp = o_stage + (c >> 1) * kChunkBytes + r * 128;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int u = (c & 1) * 4 + q;
                            *reinterpret_cast<uint4 *>(rowp + ((u ^ (r & 7)) << 4)) = w[q];
                        }
                    } else if (row_ok) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = w[q];
                    }
                }
                if (row_ok) {
                    const float lse = (m + log2f(l)) * kLn2;
                    if (p.cu_seqlens != nullptr)
                        p.lse[int64_t(h) * p.total + start + i] = lse;
                    else
                        p.lse[(int64_t(b) * p.H_row + h) * p.N + i] = lse;
                }
            }
            if (full_tile) {
                ptx::fence_proxy_async_smem();
                // every thread of the tile arrives here once, also after a
                // failed wait; the store goes out only if all 128 rows are in
                if (!ptx::bar_red_or(1 + t, 128, !ok) && r == 0) {
                    for (int ch = 0; ch < D / 64; ++ch)      // O is bf16: D / 64 chunks
                        ptx::tma_store_3d(&p.tm_o, o_stage + ch * kChunkBytes, ch * 64, h,
                                     int(start + int64_t(qt) * BM));
                    ptx::bulk_commit_and_wait_read();
                }
            }
        }
    }

    // ---- teardown ------------------------------------------------------------
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    if (warp == kWarpMma)
        ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int D, bool SPLIT>
int launch_d(const Bf16Params &p, int64_t blocks, cudaStream_t stream)
{
    auto kern = attn_fwd_bf16_kernel<D, SPLIT>;
    static PerDeviceOnce once;
    constexpr uint32_t smem = Cfg<D>::kSmemBytes;
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    if (!set_max_dynamic_smem(once, reinterpret_cast<const void *>(kern), int(smem)))
        return FA_ERR_CUDA;
    kern<<<dim3(unsigned(blocks)), dim3(kThreads), smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

namespace {
// Groups of (sequence, head) pairs for a dense, unsplit launch.  With every
// head's heaviest Q-tile pairs first, all heads' K and V are read at once;
// when they exceed what L2 holds, tiles are evicted between the Q-tile pairs
// that share them and read again from DRAM.  Past half of L2 (64 MB) the
// heads are therefore taken in consecutive groups, each small enough (about
// 32 MB of K and V) to stay in L2, as long as every group still fills the GPU
// (at least 1.5 waves of CTAs); below it one group (grouping then only adds
// the tails of the group boundaries).  1: one group.
int choose_head_groups(int bh, int n_pairs, int64_t kv_bytes_per_head)
{
    constexpr int64_t kGroupBytes = int64_t(32) << 20, kOneGroupBytes = int64_t(64) << 20;
    if (kv_bytes_per_head * bh <= kOneGroupBytes)
        return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return 1;
    int best = 1;
    for (int g = 2; g <= bh; ++g) {
        if (bh % g != 0)
            continue;
        if (2 * int64_t(n_pairs) * (bh / g) < 3 * int64_t(sms))
            break;                       // fewer CTAs per group than 1.5 waves
        best = g;
        if (kv_bytes_per_head * (bh / g) <= kGroupBytes)
            break;
    }
    return best;
}
}  // namespace

int launch_attention_bf16(const AttnArgs &a, cudaStream_t stream)
{
    Bf16Params p;
    const int Nk = a.Nk > 0 ? a.Nk : a.N;
    const int64_t total_k = a.cu_seqlens_k != nullptr ? a.total_k
                            : a.cu_seqlens != nullptr ? a.total : int64_t(a.B) * Nk;
    const int H_row = a.H_row > 0 ? a.H_row : a.H;
    if (!make_tmap_bf16(&p.tm_q, a.Q, a.total, a.H, a.d, 128, H_row) ||
        !make_tmap_bf16(&p.tm_k, a.K, total_k, a.H, a.d, 128, H_row) ||
        !make_tmap_bf16(&p.tm_v, a.V, total_k, a.H, a.d, 128, H_row) ||
        !make_tmap_bf16(&p.tm_o, a.O, a.total, a.H, a.d, 128, H_row))
        return FA_ERR_CUDA;
    p.H_row = H_row;
    p.Nk = Nk;
    p.kv_off = a.kv_off;
    p.splits = a.splits > 0 ? a.splits : 1;
    p.O_accum = a.O_accum;
    p.lse_accum = a.lse_accum;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.lse = a.lse;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    const int n_qt = (a.N + BM - 1) / BM;
    p.n_pairs = (n_qt + 1) / 2;
    p.total = a.total;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.cu_seqlens = a.cu_seqlens;
    p.cu_seqlens_k = a.cu_seqlens_k;
    p.total_k = total_k;
    p.err_word = a.err_word;
    p.expire_wait_ns = a.expire_wait_ns;
    const int64_t blocks = int64_t(p.n_pairs) * a.B * a.H * p.splits;
    if (blocks == 0)
        return FA_OK;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    const bool split = p.splits > 1 || p.kv_off != 0 || Nk != a.N || a.cu_seqlens_k != nullptr;
    // dense, unsplit launches take the heads in L2-sized groups (packed
    // batches keep one group: a late group of long sequences would be a tail)
    p.head_groups = split || a.cu_seqlens != nullptr
                        ? 1
                        : choose_head_groups(a.B * a.H, p.n_pairs, int64_t(4) * a.N * a.d);
    int rc;
    if (a.d == 64)
        rc = split ? launch_d<64, true>(p, blocks, stream) : launch_d<64, false>(p, blocks, stream);
    else
        rc = split ? launch_d<128, true>(p, blocks, stream) : launch_d<128, false>(p, blocks, stream);
    if (rc != FA_OK || p.splits == 1)
        return rc;
    return launch_attention_combine(a, stream);
}


int launch_attention_fp8(const AttnFp8Args &a, cudaStream_t stream)
{
    if (a.d != 128)
        return FA_ERR_UNSUPPORTED;
    Bf16Params p{};
    const int64_t total = a.cu_seqlens != nullptr ? a.total : int64_t(a.B) * a.N;
    if (!make_tmap_e4m3_rows(&p.tm_q, a.Qf, total, a.H, a.d) ||
        !make_tmap_e4m3_rows(&p.tm_k, a.Kf, total, a.H, a.d) ||
        !make_tmap_e4m3_vt(&p.tm_v, a.Vt, int64_t(a.B) * a.H * a.d, a.n_pad, a.d) ||
        !make_tmap_bf16(&p.tm_o, a.O, total, a.H, a.d))
        return FA_ERR_CUDA;
    p.sq = a.sq;
    p.sk = a.sk;
    p.sv = a.sv;
    p.H_row = a.H;
    p.n_tiles = (a.N + BM - 1) / BM;
    p.Nk = a.N;
    p.kv_off = 0;
    p.splits = 1;
    p.O_accum = nullptr;
    p.lse_accum = nullptr;
    p.O = static_cast<__nv_bfloat16 *>(a.O);
    p.lse = a.lse;
    p.B = a.B;
    p.H = a.H;
    p.N = a.N;
    p.n_pairs = (p.n_tiles + 1) / 2;
    p.total = total;
    p.scale_log2 = float(double(a.scale) * 1.4426950408889634);
    p.causal = a.causal;
    p.cu_seqlens = a.cu_seqlens;
    p.cu_seqlens_k = nullptr;
    p.total_k = total;
    p.err_word = a.err_word;
    p.expire_wait_ns = 0;
    const int64_t blocks = int64_t(p.n_pairs) * a.B * a.H;
    if (blocks == 0)
        return FA_OK;
    if (blocks > 0x7fffffffLL)
        return FA_ERR_TOO_LARGE;
    p.head_groups = 1;                // K' and V'^T, one byte per element, stay in L2
    auto kern = attn_fwd_bf16_kernel<128, false, true>;
    static PerDeviceOnce once;
    if (!set_max_dynamic_smem(once, reinterpret_cast<const void *>(kern),
                              int(Cfg<128, true>::kSmemBytes)))
        return FA_ERR_CUDA;
    // programmatic dependent launch of the quantisation's last kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg<128, true>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess)
        return FA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int choose_num_splits(int B, int H, int N, int Nk)
{
    // one CTA runs per SM, so the (sequence, head, Q-tile pair, split) items
    // should fill the SMs in one wave: floor(SMs / pairs) splits (a partial
    // second wave would double the time), with at least two 128-key tiles per
    // split
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    const int64_t pairs = int64_t((N + 2 * BM - 1) / (2 * BM)) * B * H;
    if (pairs <= 0 || 2 * pairs > sms)
        return 1;
    const int64_t want = sms / pairs;
    const int64_t cap = (Nk + BN - 1) / BN / 2;
    int64_t s = want < cap ? want : cap;
    if (s > 256)
        s = 256;
    return s < 1 ? 1 : int(s);
}

}  // namespace fa
