// fa_api.cu -- the extern "C" boundary of libfa.so (declared in include/fa.h):
// argument validation, stream selection, the device error word, and dispatch
// to the kernels' launchers.  No computation happens here.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "launch.h"

namespace fa {

// One copy per device that loads the library; kernels receive its address.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
thread_local cudaStream_t t_stream = nullptr;
// fa_debug_expire_next_wait: armed for the next bf16 forward or one-pass
// backward from this thread
thread_local uint32_t t_expire_wait_ns = 0;

struct DeviceInfo {
    std::once_flag once;
    int ok = 0;            // 1: compute capability 10.3 (sm_103)
    int *err_word = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

// Per-device set-up, done once with that device current.
DeviceInfo *current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    DeviceInfo *info = &g_dev[dev];
    std::call_once(info->once, [info, dev] {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess)
            return;
        info->err_word = static_cast<int *>(addr);
        info->ok = (major == 10 && minor == 3) ? 1 : 0;
    });
    return info->ok ? info : nullptr;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared validation of the attention arguments; fills `a` on success.
int check_attention(const void *Q, const void *K, const void *V, void *O, float *lse, int B, int H,
                    int N, int d, int causal, const int32_t *cu_seqlens, int64_t total,
                    bool bf16, AttnArgs *a)
{
    if (B < 0 || H < 0 || N < 0 || total < 0)
        return FA_ERR_BAD_SIZE;
    if (bf16 ? (d != 64 && d != 128) : (d < 1 || d > 128))
        return FA_ERR_UNSUPPORTED;
    if (!Q || !K || !V || !O || !lse)
        return FA_ERR_NULL_POINTER;
    const uintptr_t al = bf16 ? 16 : 4;
    if (!aligned(Q, al) || !aligned(K, al) || !aligned(V, al) || !aligned(O, al) ||
        !aligned(lse, 4))
        return FA_ERR_MISALIGNED;
    if (cu_seqlens && !aligned(cu_seqlens, 4))
        return FA_ERR_MISALIGNED;
    // TMA coordinates and the kernels' row indices are 32-bit.
    if (total > (int64_t(1) << 31) - 512 || int64_t(N) > (int64_t(1) << 31) - 512)
        return FA_ERR_TOO_LARGE;
    if (total * int64_t(H) * int64_t(d) > (int64_t(1) << 56))
        return FA_ERR_TOO_LARGE;
    a->Q = Q;
    a->K = K;
    a->V = V;
    a->O = O;
    a->lse = lse;
    a->B = B;
    a->H = H;
    a->N = N;
    a->d = d;
    a->total = total;
    a->causal = causal ? 1 : 0;
    a->cu_seqlens = cu_seqlens;
    return FA_OK;
}

// total = cu_seqlens[B], read back on the library stream (synchronises it).
int read_total(const int32_t *cu_seqlens, int B, int64_t *total)
{
    int32_t t = 0;
    if (cudaMemcpyAsync(&t, cu_seqlens + B, sizeof(t), cudaMemcpyDeviceToHost, t_stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(t_stream) != cudaSuccess)
        return FA_ERR_CUDA;
    if (t < 0)
        return FA_ERR_BAD_SIZE;
    *total = t;
    return FA_OK;
}

int attention_common(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                     int H, int N, int64_t total, bool total_known, int d, float scale,
                     int causal, const int32_t *cu_seqlens, bool bf16)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    if (B == 0 || H == 0 || N == 0)
        return FA_OK;
    DeviceInfo *dev = current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    if (cu_seqlens == nullptr) {
        total = int64_t(B) * N;
    } else if (!total_known) {
        if (!aligned(cu_seqlens, 4))
            return FA_ERR_MISALIGNED;
        const int rc = read_total(cu_seqlens, B, &total);
        if (rc != FA_OK)
            return rc;
    }
    AttnArgs a;
    const int rc = check_attention(Q, K, V, O, lse, B, H, N, d, causal, cu_seqlens, total, bf16, &a);
    if (rc != FA_OK)
        return rc;
    if (total == 0)
        return FA_OK;
    a.scale = scale;
    a.err_word = dev->err_word;
    if (!bf16)
        return launch_attention_f32(a, t_stream);
    a.expire_wait_ns = t_expire_wait_ns;
    t_expire_wait_ns = 0;
    return launch_attention_bf16(a, t_stream);
}

// Workspace of the FP8 forward: e4m3 Q', K' ([B*N, H, d]), the transposed
// V' ([B, H, d, n_pad]), then the fp32 scales; every part 256-byte aligned.
struct Fp8Layout {
    int64_t qf, kf, vt, sq, sk, vamax, sv, bytes;
    int n_tiles, n_pad;
};

// total: the rows of Q, K, V (B * N dense; the packed row count otherwise)
Fp8Layout fp8_layout(int B, int H, int N, int d, int64_t total)
{
    auto up = [](int64_t x) { return (x + 255) & ~int64_t(255); };
    Fp8Layout L;
    L.n_tiles = (N + 127) / 128;
    L.n_pad = L.n_tiles * 128;
    const int64_t elems = total * H * d;
    const int64_t tiles = int64_t(B) * H * L.n_tiles;
    int64_t off = 0;
    L.qf = off;
    off = up(off + elems);
    L.kf = off;
    off = up(off + elems);
    L.vt = off;
    off = up(off + int64_t(B) * H * d * L.n_pad);
    L.sq = off;
    off = up(off + tiles * 4);
    L.sk = off;
    off = up(off + tiles * 4);
    L.vamax = off;
    off = up(off + tiles * 4);
    L.sv = off;
    off = up(off + int64_t(B) * H * 4);
    L.bytes = off;
    return L;
}

// fa_attention_fwd_host: device copies of Q, K, V, O and lse in the caller's
// workspace, each part 256-byte aligned.
struct HostLayout {
    int64_t q, k, v, o, lse, bytes;
};

HostLayout host_layout(int B, int H, int N, int d)
{
    auto up = [](int64_t x) { return (x + 255) & ~int64_t(255); };
    const int64_t t = int64_t(B) * N * H * d * 2;
    HostLayout L;
    L.q = 0;
    L.k = L.q + up(t);
    L.v = L.k + up(t);
    L.o = L.v + up(t);
    L.lse = L.o + up(t);
    L.bytes = L.lse + up(int64_t(B) * H * N * 4);
    return L;
}

// Streams and events of the host-buffer pipeline, created once per device.
constexpr int kHostGroups = 24;   // head groups a call is cut into (at most)

// Head-group sizes of the host pipeline: about eight groups of hg = H / 8
// heads, with groups of 1, 2, 4, ... heads at both ends, so that the first
// group's copy in (before any work) and the last group's copy out (after all
// work) are short.  Returns the number of groups (sizes sum to H).
int plan_head_groups(int H, int *sizes)
{
    const int hg = (H + 7) / 8;
    int n = 0, used = 0, nd = 0, dsum = 0;
    int down[16];
    for (int s = 1; s < hg && used + s <= H && n < 8; s *= 2) {
        sizes[n++] = s;
        used += s;
    }
    for (int s = 1; s < hg && used + dsum + s <= H && nd < 8; s *= 2) {
        down[nd++] = s;
        dsum += s;
    }
    int mid = H - used - dsum;
    while (mid > 0 && n < kHostGroups - nd) {
        const int s = mid < hg ? mid : hg;
        sizes[n++] = s;
        mid -= s;
    }
    if (mid > 0) {                     // does not fit: equal groups instead
        n = 0;
        for (int h0 = 0; h0 < H; h0 += hg)
            sizes[n++] = H - h0 < hg ? H - h0 : hg;
        return n;
    }
    for (int i = nd - 1; i >= 0; --i)
        sizes[n++] = down[i];
    return n;
}
struct HostPipe {
    std::once_flag once;
    int ok = 0;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kHostGroups] = {}, comp[kHostGroups] = {};
};
HostPipe g_pipe[kMaxDevices];

HostPipe *host_pipe()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return nullptr;
    HostPipe *pp = &g_pipe[dev];
    std::call_once(pp->once, [pp] {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&pp->s_in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&pp->s_out, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&pp->start, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&pp->done, ef) != cudaSuccess)
            return;
        for (int g = 0; g < kHostGroups; ++g)
            if (cudaEventCreateWithFlags(&pp->in[g], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&pp->comp[g], ef) != cudaSuccess)
                return;
        pp->ok = 1;
    });
    return pp->ok ? pp : nullptr;
}

}  // namespace
}  // namespace fa

extern "C" {

int fa_softmax_rows(const float *x, float *y, int64_t rows, int64_t N)
{
    if (rows < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    if (rows == 0 || N == 0)
        return FA_OK;
    if (rows > (int64_t(1) << 62) / N)
        return FA_ERR_TOO_LARGE;
    if (!x || !y)
        return FA_ERR_NULL_POINTER;
    if (!fa::aligned(x, 4) || !fa::aligned(y, 4))
        return FA_ERR_MISALIGNED;
    if (fa::current_device() == nullptr)
        return FA_ERR_NO_DEVICE;
    return fa::launch_softmax_rows(x, y, rows, N, fa::t_stream);
}

int fa_attention_fwd(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                     int H, int N, int d, float scale, int causal, const int32_t *cu_seqlens)
{
    return fa::attention_common(Q, K, V, O, lse, B, H, N, 0, false, d, scale, causal, cu_seqlens,
                                true);
}

int fa_attention_fwd_varlen(const void *Q, const void *K, const void *V, void *O, float *lse,
                            int B, int H, int N, int64_t total, int d, float scale, int causal,
                            const int32_t *cu_seqlens)
{
    if (cu_seqlens == nullptr)
        return FA_ERR_NULL_POINTER;
    return fa::attention_common(Q, K, V, O, lse, B, H, N, total, true, d, scale, causal,
                                cu_seqlens, true);
}

int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (fa::current_device() == nullptr)
        return FA_ERR_NO_DEVICE;
    return fa::choose_num_splits(B, H, Nq, Nk);
}

int fa_attention_fwd_splitkv(const void *Q, const void *K, const void *V, void *O, float *lse,
                             int B, int H, int Nq, int Nk, int d, float scale, int causal,
                             int num_splits, float *O_accum, float *lse_accum)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || num_splits < 0)
        return FA_ERR_BAD_SIZE;
    if (causal && Nk < Nq)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Nq == 0)
        return FA_OK;
    if (Nk == 0)
        return FA_ERR_BAD_SIZE;            // no key for any query
    fa::DeviceInfo *dev = fa::current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    const int64_t total_q = int64_t(B) * Nq, total_k = int64_t(B) * Nk;
    if (total_k > (int64_t(1) << 31) - 512 || int64_t(Nk) > (int64_t(1) << 31) - 512)
        return FA_ERR_TOO_LARGE;
    fa::AttnArgs a;
    int rc = fa::check_attention(Q, K, V, O, lse, B, H, Nq, d, causal, nullptr, total_q, true, &a);
    if (rc != FA_OK)
        return rc;
    int splits = num_splits == 0 ? fa::choose_num_splits(B, H, Nq, Nk) : num_splits;
    const int n_kv = (Nk + 127) / 128;
    if (splits > n_kv)
        splits = n_kv;
    if (splits > 1) {
        if (O_accum == nullptr || lse_accum == nullptr)
            return FA_ERR_NULL_POINTER;
        if (!fa::aligned(O_accum, 16) || !fa::aligned(lse_accum, 4))
            return FA_ERR_MISALIGNED;
        if (int64_t(splits) * total_q * H * d > (int64_t(1) << 56))
            return FA_ERR_TOO_LARGE;
    }
    a.scale = scale;
    a.err_word = dev->err_word;
    a.Nk = Nk;
    a.kv_off = Nk - Nq;
    a.splits = splits;
    a.O_accum = splits > 1 ? O_accum : nullptr;
    a.lse_accum = splits > 1 ? lse_accum : nullptr;
    return fa::launch_attention_bf16(a, fa::t_stream);
}

}  // extern "C"

namespace fa {
namespace {
// Shared by the dense and packed backward entry points.
int attention_bwd_common(const void *Q, const void *K, const void *V, const void *O,
                         const void *dO, const float *lse, void *dQ, void *dK, void *dV,
                         float *D_buf, int B, int H, int N, int64_t total, int d, float scale,
                         int causal, const int32_t *cu_seqlens, bool one_pass = false,
                         void *workspace = nullptr, int64_t workspace_bytes = 0)
{
    if (B < 0 || H < 0 || N < 0 || total < 0 || workspace_bytes < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0 || total == 0)
        return FA_OK;
    if (!Q || !K || !V || !O || !dO || !lse || !dQ || !dK || !dV || !D_buf ||
        (one_pass && !workspace))
        return FA_ERR_NULL_POINTER;
    const void *bf[8] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void *ptr : bf)
        if (!aligned(ptr, 16))
            return FA_ERR_MISALIGNED;
    if (!aligned(lse, 4) || !aligned(D_buf, 4) || (cu_seqlens && !aligned(cu_seqlens, 4)) ||
        (one_pass && !aligned(workspace, 256)))
        return FA_ERR_MISALIGNED;
    if (total > (int64_t(1) << 31) - 512 || int64_t(N) > (int64_t(1) << 31) - 512 ||
        total * int64_t(H) * int64_t(d) > (int64_t(1) << 56))
        return FA_ERR_TOO_LARGE;
    if (one_pass && workspace_bytes < (cu_seqlens ? bwd_atomic_varlen_workspace_bytes(B, H, N, total, d)
                                                  : bwd_atomic_workspace_bytes(B, H, N, d)))
        return FA_ERR_BAD_SIZE;
    DeviceInfo *dev = current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    AttnBwdArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.dO = dO;
    a.lse = lse;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.D = D_buf;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.err_word = dev->err_word;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    if (one_pass) {
        a.dq_acc = static_cast<float *>(workspace);
        a.expire_wait_ns = t_expire_wait_ns;
        t_expire_wait_ns = 0;
        return launch_attention_bwd_atomic(a, t_stream);
    }
    return launch_attention_bwd(a, t_stream);
}
}  // namespace
}  // namespace fa

extern "C" {

int fa_attention_fwd_splitkv_varlen(const void *Q, const void *K, const void *V, void *O,
                                    float *lse, int B, int H, int Nq, int Nk, int64_t total_q,
                                    int64_t total_k, int d, float scale, int causal,
                                    int num_splits, const int32_t *cu_seqlens_q,
                                    const int32_t *cu_seqlens_k, float *O_accum,
                                    float *lse_accum)
{
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || total_q < 0 || total_k < 0 || num_splits < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (cu_seqlens_q == nullptr || cu_seqlens_k == nullptr)
        return FA_ERR_NULL_POINTER;
    if (B == 0 || H == 0 || Nq == 0 || total_q == 0)
        return FA_OK;
    if (Nk == 0 || total_k == 0)
        return FA_ERR_BAD_SIZE;            // no key for any query
    fa::DeviceInfo *dev = fa::current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    if (total_k > (int64_t(1) << 31) - 512 || int64_t(Nk) > (int64_t(1) << 31) - 512)
        return FA_ERR_TOO_LARGE;
    if (!fa::aligned(cu_seqlens_k, 4))
        return FA_ERR_MISALIGNED;
    fa::AttnArgs a;
    int rc = fa::check_attention(Q, K, V, O, lse, B, H, Nq, d, causal, cu_seqlens_q, total_q, true,
                                 &a);
    if (rc != FA_OK)
        return rc;
    int splits = num_splits == 0 ? fa::choose_num_splits(B, H, Nq, Nk) : num_splits;
    const int n_kv = (Nk + 127) / 128;
    if (splits > n_kv)
        splits = n_kv;
    if (splits > 1) {
        if (O_accum == nullptr || lse_accum == nullptr)
            return FA_ERR_NULL_POINTER;
        if (!fa::aligned(O_accum, 16) || !fa::aligned(lse_accum, 4))
            return FA_ERR_MISALIGNED;
        if (int64_t(splits) * total_q * H * d > (int64_t(1) << 56))
            return FA_ERR_TOO_LARGE;
    }
    a.scale = scale;
    a.err_word = dev->err_word;
    a.Nk = Nk;
    a.kv_off = 0;                          // per sequence, from the two prefix sums
    a.splits = splits;
    a.O_accum = splits > 1 ? O_accum : nullptr;
    a.lse_accum = splits > 1 ? lse_accum : nullptr;
    a.cu_seqlens_k = cu_seqlens_k;
    a.total_k = total_k;
    return fa::launch_attention_bf16(a, fa::t_stream);
}

int fa_attention_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                     const float *lse, void *dQ, void *dK, void *dV, float *D_buf, int B, int H,
                     int N, int d, float scale, int causal)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    return fa::attention_bwd_common(Q, K, V, O, dO, lse, dQ, dK, dV, D_buf, B, H, N,
                                    int64_t(B) * N, d, scale, causal, nullptr);
}

int fa_attention_bwd_varlen(const void *Q, const void *K, const void *V, const void *O,
                            const void *dO, const float *lse, void *dQ, void *dK, void *dV,
                            float *D_buf, int B, int H, int N, int64_t total, int d, float scale,
                            int causal, const int32_t *cu_seqlens)
{
    if (cu_seqlens == nullptr)
        return FA_ERR_NULL_POINTER;
    return fa::attention_bwd_common(Q, K, V, O, dO, lse, dQ, dK, dV, D_buf, B, H, N, total, d,
                                    scale, causal, cu_seqlens);
}

int fa_attention_bwd_atomic(const void *Q, const void *K, const void *V, const void *O,
                            const void *dO, const float *lse, void *dQ, void *dK, void *dV,
                            float *D_buf, int B, int H, int N, int d, float scale, int causal,
                            void *workspace, int64_t workspace_bytes)
{
    return fa::attention_bwd_common(Q, K, V, O, dO, lse, dQ, dK, dV, D_buf, B, H, N,
                                    int64_t(B) * N, d, scale, causal, nullptr, true, workspace,
                                    workspace_bytes);
}

int fa_attention_bwd_atomic_varlen(const void *Q, const void *K, const void *V, const void *O,
                                   const void *dO, const float *lse, void *dQ, void *dK,
                                   void *dV, float *D_buf, int B, int H, int N, int64_t total,
                                   int d, float scale, int causal, const int32_t *cu_seqlens,
                                   void *workspace, int64_t workspace_bytes)
{
    if (cu_seqlens == nullptr)
        return FA_ERR_NULL_POINTER;
    return fa::attention_bwd_common(Q, K, V, O, dO, lse, dQ, dK, dV, D_buf, B, H, N, total, d,
                                    scale, causal, cu_seqlens, true, workspace, workspace_bytes);
}

int64_t fa_attention_bwd_atomic_varlen_workspace_bytes(int B, int H, int N, int64_t total, int d)
{
    if (B < 0 || H < 0 || N < 0 || total < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    return fa::bwd_atomic_varlen_workspace_bytes(B, H, N, total, d);
}

int64_t fa_attention_bwd_atomic_workspace_bytes(int B, int H, int N, int d)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    return fa::bwd_atomic_workspace_bytes(B, H, N, d);
}

}  // extern "C"

namespace fa {
namespace {
// Shared by the dense and packed FP8 entry points.
int attention_fp8_common(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                         int H, int N, int64_t total, int d, float scale, int causal,
                         const int32_t *cu_seqlens, const float *signs, void *workspace,
                         int64_t workspace_bytes)
{
    if (B < 0 || H < 0 || N < 0 || total < 0 || workspace_bytes < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 128)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0 || total == 0)
        return FA_OK;
    if (!Q || !K || !V || !O || !lse || !signs || !workspace)
        return FA_ERR_NULL_POINTER;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) ||
        !aligned(lse, 4) || !aligned(signs, 4) || !aligned(workspace, 256) ||
        (cu_seqlens && !aligned(cu_seqlens, 4)))
        return FA_ERR_MISALIGNED;
    if (total > (int64_t(1) << 31) - 512 || int64_t(N) > (int64_t(1) << 31) - 512 ||
        total * int64_t(H) * int64_t(d) > (int64_t(1) << 56))
        return FA_ERR_TOO_LARGE;
    const Fp8Layout L = fp8_layout(B, H, N, d, total);
    if (workspace_bytes < L.bytes)
        return FA_ERR_BAD_SIZE;
    DeviceInfo *dev = current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Fp8QuantArgs q;
    q.Q = Q;
    q.K = K;
    q.V = V;
    q.signs = signs;
    q.Qf = ws + L.qf;
    q.Kf = ws + L.kf;
    q.Vt = ws + L.vt;
    q.sq = reinterpret_cast<float *>(ws + L.sq);
    q.sk = reinterpret_cast<float *>(ws + L.sk);
    q.vamax = reinterpret_cast<float *>(ws + L.vamax);
    q.sv = reinterpret_cast<float *>(ws + L.sv);
    q.B = B;
    q.H = H;
    q.N = N;
    q.d = d;
    q.err_word = dev->err_word;
    q.cu_seqlens = cu_seqlens;
    q.total = total;
    int rc = launch_fp8_quantize(q, t_stream);
    if (rc != FA_OK)
        return rc;
    AttnFp8Args a;
    a.Qf = q.Qf;
    a.Kf = q.Kf;
    a.Vt = q.Vt;
    a.sq = q.sq;
    a.sk = q.sk;
    a.sv = q.sv;
    a.O = O;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.n_pad = L.n_pad;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.err_word = dev->err_word;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    return launch_attention_fp8(a, t_stream);
}
}  // namespace
}  // namespace fa

extern "C" {

int64_t fa_attention_fp8_workspace_bytes(int B, int H, int N, int d)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 128)
        return FA_ERR_UNSUPPORTED;
    return fa::fp8_layout(B, H, N, d, int64_t(B) * N).bytes;
}

int64_t fa_attention_fp8_varlen_workspace_bytes(int B, int H, int N, int64_t total, int d)
{
    if (B < 0 || H < 0 || N < 0 || total < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 128)
        return FA_ERR_UNSUPPORTED;
    return fa::fp8_layout(B, H, N, d, total).bytes;
}

int fa_attention_fwd_fp8(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                         int H, int N, int d, float scale, int causal, const float *signs,
                         void *workspace, int64_t workspace_bytes)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    return fa::attention_fp8_common(Q, K, V, O, lse, B, H, N, int64_t(B) * N, d, scale, causal,
                                    nullptr, signs, workspace, workspace_bytes);
}

int fa_attention_fwd_fp8_varlen(const void *Q, const void *K, const void *V, void *O, float *lse,
                                int B, int H, int N, int64_t total, int d, float scale,
                                int causal, const int32_t *cu_seqlens, const float *signs,
                                void *workspace, int64_t workspace_bytes)
{
    if (cu_seqlens == nullptr)
        return FA_ERR_NULL_POINTER;
    return fa::attention_fp8_common(Q, K, V, O, lse, B, H, N, total, d, scale, causal,
                                    cu_seqlens, signs, workspace, workspace_bytes);
}

int64_t fa_attention_host_workspace_bytes(int B, int H, int N, int d)
{
    if (B < 0 || H < 0 || N < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    return fa::host_layout(B, H, N, d).bytes;
}

int fa_attention_fwd_host(const void *Q, const void *K, const void *V, void *O, float *lse, int B,
                          int H, int N, int d, float scale, int causal, void *workspace,
                          int64_t workspace_bytes)
{
    if (B < 0 || H < 0 || N < 0 || workspace_bytes < 0)
        return FA_ERR_BAD_SIZE;
    if (d != 64 && d != 128)
        return FA_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0)
        return FA_OK;
    if (!Q || !K || !V || !O || !lse || !workspace)
        return FA_ERR_NULL_POINTER;
    if (!fa::aligned(workspace, 256))
        return FA_ERR_MISALIGNED;
    const int64_t total = int64_t(B) * N;
    if (total > (int64_t(1) << 31) - 512 || total * int64_t(H) * int64_t(d) > (int64_t(1) << 56))
        return FA_ERR_TOO_LARGE;
    const fa::HostLayout L = fa::host_layout(B, H, N, d);
    if (workspace_bytes < L.bytes)
        return FA_ERR_BAD_SIZE;
    fa::DeviceInfo *dev = fa::current_device();
    if (dev == nullptr)
        return FA_ERR_NO_DEVICE;
    fa::HostPipe *pp = fa::host_pipe();
    if (pp == nullptr)
        return FA_ERR_CUDA;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *dq = ws + L.q, *dk = ws + L.k, *dv = ws + L.v, *dout = ws + L.o;
    float *dl = reinterpret_cast<float *>(ws + L.lse);
    const uint8_t *hq = static_cast<const uint8_t *>(Q), *hk = static_cast<const uint8_t *>(K),
                  *hv = static_cast<const uint8_t *>(V);
    uint8_t *ho = static_cast<uint8_t *>(O);
    // head groups; a group's slice of a token row is hn * d * 2 contiguous
    // bytes of the row's H * d * 2
    int sizes[fa::kHostGroups];
    const int n_groups = fa::plan_head_groups(H, sizes);
    const size_t row = size_t(H) * d * 2, lse_row = size_t(H) * N * 4;
    const cudaStream_t s_main = fa::t_stream;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    // Every group's arguments are checked before anything is enqueued.
    fa::AttnArgs args[fa::kHostGroups];
    for (int g = 0, h0 = 0; g < n_groups; h0 += sizes[g], ++g) {
        const size_t off = size_t(h0) * d * 2;
        const int rc = fa::check_attention(dq + off, dk + off, dv + off, dout + off,
                                           dl + size_t(h0) * N, B, sizes[g], N, d, causal,
                                           nullptr, total, true, &args[g]);
        if (rc != FA_OK)
            return rc;
        args[g].H_row = H;
        args[g].scale = scale;
        args[g].err_word = dev->err_word;
    }
    // On a failure after the first copy is enqueued, the library stream still
    // waits for both helper streams, so the copies that read the caller's
    // host buffers are ordered before anything the caller synchronises on.
    auto join_and_fail = [&](int rc) {
        if (cudaEventRecord(pp->done, pp->s_in) == cudaSuccess)
            cudaStreamWaitEvent(s_main, pp->done, 0);
        if (cudaEventRecord(pp->done, pp->s_out) == cudaSuccess)
            cudaStreamWaitEvent(s_main, pp->done, 0);
        return rc;
    };
    if (!ok(cudaEventRecord(pp->start, s_main)) || !ok(cudaStreamWaitEvent(pp->s_in, pp->start, 0)) ||
        !ok(cudaStreamWaitEvent(pp->s_out, pp->start, 0)))
        return join_and_fail(FA_ERR_CUDA);
    for (int g = 0, h0 = 0; g < n_groups; h0 += sizes[g], ++g) {
        const int hn = sizes[g];
        const size_t off = size_t(h0) * d * 2, width = size_t(hn) * d * 2;
        if (!ok(cudaMemcpy2DAsync(dq + off, row, hq + off, row, width, size_t(total),
                                  cudaMemcpyHostToDevice, pp->s_in)) ||
            !ok(cudaMemcpy2DAsync(dk + off, row, hk + off, row, width, size_t(total),
                                  cudaMemcpyHostToDevice, pp->s_in)) ||
            !ok(cudaMemcpy2DAsync(dv + off, row, hv + off, row, width, size_t(total),
                                  cudaMemcpyHostToDevice, pp->s_in)) ||
            !ok(cudaEventRecord(pp->in[g], pp->s_in)) ||
            !ok(cudaStreamWaitEvent(s_main, pp->in[g], 0)))
            return join_and_fail(FA_ERR_CUDA);
        const int rc = fa::launch_attention_bf16(args[g], s_main);
        if (rc != FA_OK)
            return join_and_fail(rc);
        if (!ok(cudaEventRecord(pp->comp[g], s_main)) ||
            !ok(cudaStreamWaitEvent(pp->s_out, pp->comp[g], 0)) ||
            !ok(cudaMemcpy2DAsync(ho + off, row, dout + off, row, width, size_t(total),
                                  cudaMemcpyDeviceToHost, pp->s_out)) ||
            !ok(cudaMemcpy2DAsync(lse + size_t(h0) * N, lse_row, dl + size_t(h0) * N, lse_row,
                                  size_t(hn) * N * 4, size_t(B), cudaMemcpyDeviceToHost,
                                  pp->s_out)))
            return join_and_fail(FA_ERR_CUDA);
    }
    if (!ok(cudaEventRecord(pp->done, pp->s_out)) || !ok(cudaStreamWaitEvent(s_main, pp->done, 0)))
        return join_and_fail(FA_ERR_CUDA);
    return FA_OK;
}

int fa_attention_fwd_f32(const float *Q, const float *K, const float *V, float *O, float *lse,
                         int B, int H, int N, int d, float scale, int causal,
                         const int32_t *cu_seqlens)
{
    return fa::attention_common(Q, K, V, O, lse, B, H, N, 0, false, d, scale, causal, cu_seqlens,
                                false);
}

int fa_debug_expire_next_wait(int64_t ns)
{
    if (ns < 0 || ns > 1000000000)
        return FA_ERR_BAD_SIZE;
    fa::t_expire_wait_ns = uint32_t(ns);
    return FA_OK;
}

int fa_set_stream(void *stream)
{
    fa::t_stream = static_cast<cudaStream_t>(stream);
    return FA_OK;
}

void *fa_get_stream(void) { return fa::t_stream; }

int fa_get_device_error(void)
{
    if (fa::current_device() == nullptr)
        return FA_ERR_NO_DEVICE;
    int v = 0;
    const int zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, fa::g_device_error, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(fa::g_device_error, &zero, sizeof(zero)) != cudaSuccess)
        return FA_ERR_CUDA;
    return v;
}

const char *fa_strerror(int code)
{
    switch (code) {
    case FA_OK: return "success";
    case FA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case FA_ERR_BAD_SIZE: return "a size is negative or inconsistent";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or option";
    case FA_ERR_MISALIGNED: return "a pointer breaks the alignment rule";
    case FA_ERR_CUDA: return "a CUDA call failed";
    case FA_ERR_TOO_LARGE: return "a size exceeds what the kernels can index";
    case FA_ERR_NO_DEVICE: return "no sm_103 device is current";
    case FA_ERR_SCRATCH_LIMIT:
        return "the problem needs more scratch than the library's static array holds";
    default: return "unknown error code";
    }
}

int fa_version(void) { return 100; }

}  // extern "C"
