"""The C-ABI library builds, loads and exports what include/fa.h declares (no GPU).

Also checks the host-side argument validation that returns before any CUDA
call (negative sizes, empty work).  No kernel is launched here.
"""
import ctypes
import os
import re

import pytest

import online_softmax_06_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.lib()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa_softmax_rows", "fa_attention_fwd", "fa_attention_fwd_f32",
                     "fa_attention_fwd_varlen", "fa_set_stream", "fa_get_device_error",
                     "fa_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_only_the_boundary_is_exported():
    # -fvisibility=hidden: the kernels' host launchers stay internal
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in exported if s.startswith("fa_")}
    assert ours == set(declared_functions())


def test_version_and_strerror(lib):
    assert fa.fa_version() >= 100
    assert fa.strerror(0) == "success"
    assert "NULL" in fa.strerror(-1)
    assert fa.strerror(12345) == "unknown error code"


def test_host_validation_without_gpu(lib):
    # these return before any CUDA call
    assert fa.fa_softmax_rows(None, None, -1, 4) == -2
    assert fa.fa_softmax_rows(None, None, 0, 4) == 0
    assert fa.fa_softmax_rows(None, None, 4, 0) == 0
    assert fa.fa_attention_fwd(None, None, None, None, None, -1, 1, 1, 64, 1.0, 0, None) == -2
    assert fa.fa_attention_fwd(None, None, None, None, None, 0, 1, 1, 64, 1.0, 0, None) == 0
    assert fa.fa_attention_fwd_varlen(None, None, None, None, None, 1, 1, 1, 1, 64, 1.0, 0,
                                      None) == -1
    assert fa.fa_attention_fwd_f32(None, None, None, None, None, 1, -1, 1, 64, 1.0, 0, None) == -2
    assert fa.fa_attention_bwd(None, None, None, None, None, None, None, None, None, None,
                               1, 1, -1, 64, 1.0, 0) == -2
    assert fa.fa_attention_bwd(None, None, None, None, None, None, None, None, None, None,
                               1, 1, 8, 80, 1.0, 0) == -3
    assert fa.fa_attention_bwd(None, None, None, None, None, None, None, None, None, None,
                               0, 1, 8, 64, 1.0, 0) == 0
    assert fa.fa_attention_bwd(None, None, None, None, None, None, None, None, None, None,
                               1, 1, 8, 64, 1.0, 0) == -1
    hw = fa.fa_attention_host_workspace_bytes
    assert hw(-1, 1, 1, 64) == -2
    assert hw(1, 1, 1, 96) == -3
    # four bf16 [2, 5, 3, 64] tensors (3840 bytes each) and lse [2, 3, 5] fp32,
    # every part rounded up to 256 bytes
    assert hw(2, 3, 5, 64) == 4 * 3840 + 256
    fh = fa.fa_attention_fwd_host
    assert fh(None, None, None, None, None, -1, 1, 1, 64, 1.0, 0, None, 0) == -2
    assert fh(None, None, None, None, None, 1, 1, 1, 96, 1.0, 0, None, 0) == -3
    assert fh(None, None, None, None, None, 0, 1, 1, 64, 1.0, 0, None, 0) == 0
    assert fh(None, None, None, None, None, 1, 1, 1, 64, 1.0, 0, None, 0) == -1
    assert fh(16, 16, 16, 16, 16, 1, 1, 1, 64, 1.0, 0, 8, 1 << 20) == -4      # workspace alignment
    assert fh(16, 16, 16, 16, 16, 1, 1, 1, 64, 1.0, 0, 256, 1) == -2          # workspace size
    nl = fa.fa_attention_fwd_splitkv_noalloc
    assert nl(None, None, None, None, None, 1, 1, -1, 8, 64, 1.0, 0, 0) == -2
    assert nl(None, None, None, None, None, 1, 1, 9, 8, 64, 1.0, 1, 0) == -2   # causal Nk < Nq
    assert nl(None, None, None, None, None, 1, 1, 8, 8, 96, 1.0, 0, 0) == -3
    assert nl(None, None, None, None, None, 0, 1, 8, 8, 64, 1.0, 0, 0) == 0


def test_one_pass_backward_host_checks_without_gpu(lib):
    """The one-pass backward's workspace sizes and its argument checks that
    return before any CUDA call."""
    wb = fa.fa_attention_bwd_atomic_workspace_bytes
    assert wb(-1, 1, 8, 128) == fa.FA_ERR_BAD_SIZE
    assert wb(1, 1, 8, 96) == fa.FA_ERR_UNSUPPORTED
    # accumulator [B H, n_pad, d] fp32 and (lse, D) pairs [B H, n_pad], n_pad = 64
    assert wb(2, 3, 50, 128) == 2 * 3 * 64 * (128 + 2) * 4
    assert wb(2, 3, 50, 64) == 2 * 3 * 64 * (64 + 2) * 4
    assert wb(2, 3, 64, 128) == wb(2, 3, 50, 128)
    assert wb(2, 3, 65, 128) == 2 * 3 * 128 * (128 + 2) * 4
    vb = fa.fa_attention_bwd_atomic_varlen_workspace_bytes
    assert vb(2, 3, 50, -1, 128) == fa.FA_ERR_BAD_SIZE
    assert vb(2, 3, 50, 90, 96) == fa.FA_ERR_UNSUPPORTED
    # accumulator [H, total + 64, d] fp32 and pairs [H, B, n_pad]
    assert vb(2, 3, 50, 90, 128) == 3 * (90 + 64) * 128 * 4 + 3 * 2 * 64 * 8
    assert vb(2, 3, 50, 90, 64) == 3 * (90 + 64) * 64 * 4 + 3 * 2 * 64 * 8
    call = fa.fa_attention_bwd_atomic
    p = [None] * 10
    assert call(*p, 1, 1, -1, 128, 1.0, 0, None, 0) == fa.FA_ERR_BAD_SIZE
    assert call(*p, 1, 1, 8, 96, 1.0, 0, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert call(*p, 0, 1, 8, 128, 1.0, 0, None, 0) == 0
    assert call(*p, 1, 1, 8, 128, 1.0, 0, None, 0) == fa.FA_ERR_NULL_POINTER
    assert call(*p, 1, 1, 8, 128, 1.0, 0, None, -1) == fa.FA_ERR_BAD_SIZE
    ptrs = [256] * 10
    assert call(*ptrs, 1, 1, 8, 128, 1.0, 0, 16, 1 << 20) == fa.FA_ERR_MISALIGNED
    assert call(*ptrs, 1, 1, 8, 128, 1.0, 0, 256, wb(1, 1, 8, 128) - 4) == fa.FA_ERR_BAD_SIZE
    vcall = fa.fa_attention_bwd_atomic_varlen
    assert vcall(*p, 1, 1, 8, 8, 128, 1.0, 0, None, None, 0) == fa.FA_ERR_NULL_POINTER
    assert vcall(*ptrs, 1, 1, 8, 8, 128, 1.0, 0, 256, 256,
                 vb(1, 1, 8, 8, 128) - 8) == fa.FA_ERR_BAD_SIZE


def test_expire_wait_argument_range(lib):
    """The failure-detection switch takes 0 (off) .. 10^9 ns and is checked on
    the host (no device needed)."""
    assert fa.fa_debug_expire_next_wait(-1) == fa.FA_ERR_BAD_SIZE
    assert fa.fa_debug_expire_next_wait(10**9 + 1) == fa.FA_ERR_BAD_SIZE
    assert fa.fa_debug_expire_next_wait(0) == 0


def test_noalloc_scratch_size_matches_header():
    text = open(HEADER, encoding="utf-8").read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m, "FA_NOALLOC_SCRATCH_BYTES not found"
    assert int(m[1]) * int(m[2]) * int(m[3]) == fa.FA_NOALLOC_SCRATCH_BYTES
    assert re.search(r"#define FA_ERR_SCRATCH_LIMIT \((-\d+)\)", text)[1] == \
        str(fa.FA_ERR_SCRATCH_LIMIT)


def test_stream_setting_is_per_thread(lib):
    import threading
    fa.fa_set_stream(ctypes.c_void_p(0x1234))
    seen = []
    t = threading.Thread(target=lambda: seen.append(fa.fa_get_stream()))
    t.start()
    t.join()
    assert fa.fa_get_stream() == 0x1234
    assert seen == [None]
    fa.fa_set_stream(None)
    assert fa.fa_get_stream() is None


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="CPU-only check")
def test_no_device_is_reported(lib):
    # valid-looking sizes with no GPU present: the library refuses before launching
    assert fa.fa_softmax_rows(ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 4) == -7


def test_tensor_wrappers_refuse_host_tensors():
    """No CPU fallback: the device-tensor wrappers reject host tensors before
    anything runs (the host-buffer entry point is the one that takes them)."""
    import torch
    import online_softmax_06_gb300 as fa
    x = torch.zeros((4, 8), dtype=torch.float32)
    q = torch.zeros((1, 8, 1, 64), dtype=torch.bfloat16)
    lse = torch.zeros((1, 1, 8), dtype=torch.float32)
    signs = torch.ones(128, dtype=torch.float32)
    q128 = torch.zeros((1, 8, 1, 128), dtype=torch.bfloat16)
    calls = [
        lambda: fa.softmax_rows(x),
        lambda: fa.attention_fwd(q, q, q),
        lambda: fa.attention_fwd(q.float(), q.float(), q.float()),
        lambda: fa.attention_fwd_splitkv(q, q, q),
        lambda: fa.attention_fwd_fp8(q128, q128, q128, signs),
        lambda: fa.attention_bwd(q, q, q, q, q, lse),
    ]
    for call in calls:
        with pytest.raises(ValueError):
            call()
