"""The C ABI on a machine without a GPU: the library loads, exports every
entry point include/ssd.h declares, and rejects bad arguments on the host
before touching CUDA."""
import ctypes
import os
import re

import pytest

import mamba_ssd_chunked_gb300 as pkg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from mamba_ssd_chunked_gb300 import build
    build.build()
    return pkg.library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ssd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"SSD_API\s+[\w\s\*]+?\b(ssd_\w+)\s*\(", text)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ("ssd_fwd", "ssd_fwd_ws", "ssd_fwd_host", "ssd_fwd_workspace_bytes", "ssd_device_status",
              "ssd_status_string", "ssd_kernel_launches", "ssd_release", "ssd_select_path", "ssd_step",
              "ssd_conv1d_silu", "ssd_conv1d_step", "ssd_gated_rmsnorm", "ssd_fwd_ex", "ssd_step_ex",
              "ssd_debug_build", "ssd_debug_failed_line", "ssd_check_inputs", "ssd_host_slices"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libssd.so does not export {name}"


def test_kernel_timing_arguments(lib):
    import ctypes
    lib.ssd_kernel_timing(0)
    assert lib.ssd_kernel_timing_read(None, None) == 1  # SSD_ERR_INVALID_ARG
    ms, n = ctypes.c_double(-1.0), ctypes.c_uint64(7)
    assert lib.ssd_kernel_timing_read(ctypes.byref(ms), ctypes.byref(n)) == 0  # nothing recorded: no CUDA call
    assert ms.value == 0.0 and n.value == 0


def test_release_and_debug_builds_say_which_they_are(lib):
    import ctypes as ct
    from mamba_ssd_chunked_gb300 import build
    assert lib.ssd_debug_build() == 0
    dbg = ct.CDLL(build.build(debug=True))
    assert dbg.ssd_debug_build() == 1
    names = declared_functions()
    for name in names:
        assert hasattr(dbg, name), f"libssd_debug.so does not export {name}"


def test_status_strings(lib):
    for code in range(7):
        assert lib.ssd_status_string(code)
    assert lib.ssd_status_string(99) == b"unknown status"


def _dims(**kw):
    base = dict(batch=2, seqlen=300, nheads=4, headdim=64, ngroups=2, dstate=128)
    base.update(kw)
    return pkg.Dims(*[base[k] for k in ("batch", "seqlen", "nheads", "headdim", "ngroups", "dstate")])


# Every pointer handed to the library below is a real, writable buffer of at
# least the size the call declares (host memory: this file runs without a
# GPU). Validation rejects each call before any CUDA work; if that ever
# changed, the damage would be a wrong return code or output, not a fault.
_BUF = ctypes.create_string_buffer(8 << 20)
FAKE = (ctypes.addressof(_BUF) + 15) // 16 * 16  # 16-byte aligned
assert FAKE + 4 * 1024 * 1024 <= ctypes.addressof(_BUF) + len(_BUF)


@pytest.mark.parametrize("bad", [
    dict(batch=0), dict(seqlen=0), dict(nheads=0), dict(headdim=0), dict(dstate=0), dict(ngroups=0),
    dict(nheads=6, ngroups=4),
])
def test_bad_dims_rejected_on_host(lib, bad):
    d = _dims(**bad)
    rc = lib.ssd_fwd(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, d.ngroups, FAKE,
                     None, None)
    assert rc == 1


def test_null_required_pointer_rejected(lib):
    d = _dims()
    rc = lib.ssd_fwd(ctypes.byref(d), 1, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, FAKE, None, None)
    assert rc == 1
    rc = lib.ssd_fwd(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, None, None, None)
    assert rc == 1


def test_ngroups_argument_must_match_dims(lib):
    d = _dims()
    rc = lib.ssd_fwd(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 1, FAKE, None, None)
    assert rc == 1


def test_bad_dtype_and_chunk_rejected(lib):
    d = _dims()
    assert lib.ssd_fwd(ctypes.byref(d), 7, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, FAKE, None,
                       None) == 1
    assert lib.ssd_fwd(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 0, 2, FAKE, None,
                       None) == 1


def test_misaligned_pointer_is_unsupported(lib):
    d = _dims()
    rc = lib.ssd_fwd(ctypes.byref(d), 1, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, FAKE, None,
                     None)
    assert rc == 2


def test_unsupported_chunk_len(lib):
    d = _dims()
    rc = lib.ssd_fwd(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 512, 2, FAKE, None, None)
    assert rc == 2
    rc = lib.ssd_fwd_ws(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 64, 2, FAKE, None, 2,
                        FAKE, 4 << 20, None)
    assert rc == 2  # the tensor-core path takes chunk_len 128 or 256 only


def test_workspace_too_small(lib):
    d = _dims()
    need = lib.ssd_fwd_workspace_bytes(ctypes.byref(d), 1, 256, 2)
    assert 0 < need and need + 64 <= 4 << 20
    rc = lib.ssd_fwd_ws(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, FAKE, None, 2,
                        FAKE, need - 1, None)
    assert rc == 5
    rc = lib.ssd_fwd_ws(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 2, FAKE, None, 2,
                        FAKE + 16, need + 64, None)
    assert rc == 5  # not 256-byte aligned


def test_path_selection(lib):
    assert pkg.ssd_select_path(4, 4096, 80, 64, 1, 128, "bf16", 256) == "chain"
    assert pkg.ssd_select_path(4, 4096, 80, 64, 1, 128, "bf16", 128) == "chain"
    assert pkg.ssd_select_path(1, 131072, 64, 64, 1, 256, "bf16", 256) == "chain"  # dstate 256
    assert pkg.ssd_select_path(1, 4096, 6, 64, 2, 128, "bf16", 256) == "tc"  # odd heads per group
    assert pkg.ssd_select_path(1, 4096, 6, 64, 2, 256, "bf16", 256) == "tc"
    assert pkg.ssd_select_path(1, 4096, 4, 64, 1, 192, "bf16", 256) == "simt"  # dstate neither 128 nor 256
    assert pkg.ssd_select_path(1, 256, 4, 16, 1, 16, "f32", 64) == "simt"
    assert pkg.ssd_select_path(4, 4096, 80, 64, 1, 128, "f32", 256) == "simt"
    assert pkg.ssd_select_path(4, 4096, 80, 32, 1, 128, "bf16", 256) == "simt"
    assert pkg.ssd_select_path(2, 4096, 40, 128, 1, 128, "bf16", 256) == "chain"  # headdim 128: a chain per head
    assert pkg.ssd_select_path(1, 4096, 5, 128, 5, 256, "bf16", 256) == "chain"  # odd heads per group are fine
    assert pkg.ssd_select_path(2, 4096, 40, 128, 1, 128, "f32", 256) == "simt"
    assert pkg.ssd_select_path(4, 4096, 80, 64, 1, 128, "bf16", 64) == "simt"


def visible_sm_count() -> int:
    """SM count of the current CUDA device, 0 where none is visible."""
    try:
        import torch
    except ImportError:
        return 0
    if not torch.cuda.is_available():
        return 0
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def test_workspace_sizes(lib):
    # tensor-core path: a work counter, two ready flags per (batch, head) and
    # two fp32 state slots per (batch, head)
    b, h, p, n = 4, 80, 64, 128
    need = pkg.ssd_fwd_workspace_bytes(b, 4096, h, p, 1, n, "bf16", 256, "tc")
    slots = 4 * b * h * 2 * p * n
    counters = 4 * (1 + 2 * b * h)
    assert slots + counters <= need <= slots + counters + 4096
    # SIMT path: one fp32 state per chunk
    need = pkg.ssd_fwd_workspace_bytes(1, 256, 4, 16, 1, 16, "f32", 64, "simt")
    assert need >= 4 * 1 * 4 * 4 * 16 * 16
    assert pkg.ssd_fwd_workspace_bytes(1, 256, 4, 16, 1, 16, "f32", 64, "tc") == 0
    # chain path: a counter and flag per CTA, one hand-off state per CTA (two
    # heads), one CTA per SM; without a device to ask for its SM count it sizes
    # for 1024 CTAs
    ncta = min(visible_sm_count() or 1024, b * (h // 2) * 16)
    need = pkg.ssd_fwd_workspace_bytes(b, 4096, h, p, 1, n, "bf16", 256, "chain")
    assert need >= ncta * 2 * p * n * 4
    need256 = pkg.ssd_fwd_workspace_bytes(b, 4096, h, p, 1, 256, "bf16", 256, "chain")
    assert need256 >= ncta * 2 * p * 256 * 4  # the hand-off states are twice as wide
    assert need256 - need >= ncta * 2 * p * 128 * 4
    assert pkg.ssd_fwd_workspace_bytes(b, 4096, h, p, 1, 192, "bf16", 256, "chain") == 0


def test_kernel_counter_starts_without_launches(lib):
    assert lib.ssd_kernel_launches() >= 0


def test_step_rejects_bad_arguments_on_host(lib):
    d = pkg.Dims(2, 2, 4, 64, 2, 128)   # seqlen must be 1
    assert lib.ssd_step(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, FAKE, None) == 1
    d = pkg.Dims(2, 1, 4, 64, 2, 128)
    assert lib.ssd_step(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 2, FAKE, None) == 1
    assert lib.ssd_step(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, FAKE, None) == 1
    assert lib.ssd_step(ctypes.byref(d), 1, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 2, FAKE, None) == 2


def test_conv_rejects_bad_arguments_on_host(lib):
    d = pkg.ConvDims(2, 16, 64, 1, 16, 4)           # conv_dim = 96
    call = lib.ssd_conv1d_silu
    assert call(None, 1, FAKE, 96, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 1
    assert call(ctypes.byref(d), 1, None, 96, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 1
    assert call(ctypes.byref(d), 1, FAKE, 95, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 1   # stride < conv_dim
    assert call(ctypes.byref(d), 3, FAKE, 96, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 1   # dtype
    big = pkg.ConvDims(2, 16, 64, 1, 16, 9)          # more than 8 taps
    assert call(ctypes.byref(big), 1, FAKE, 96, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 2
    assert call(ctypes.byref(d), 1, FAKE + 1, 96, FAKE, None, 1, FAKE, FAKE, FAKE, None, None) == 2  # misaligned
    assert lib.ssd_conv1d_step(ctypes.byref(d), 1, FAKE, 96, FAKE, None, 1, FAKE, FAKE, FAKE, FAKE, None) == 1
    one = pkg.ConvDims(2, 1, 64, 1, 16, 4)
    assert lib.ssd_conv1d_step(ctypes.byref(one), 1, FAKE, 96, FAKE, None, 1, None, FAKE, FAKE, FAKE, None) == 1


def test_norm_rejects_bad_arguments_on_host(lib):
    f = lib.ssd_gated_rmsnorm
    assert f(1, 4, 64, 0, None, 64, None, 0, FAKE, 1e-5, FAKE, 64, None) == 1            # y NULL
    assert f(1, 4, 64, 0, FAKE, 63, None, 0, FAKE, 1e-5, FAKE, 64, None) == 1            # stride < dim
    assert f(1, 4, 64, 24, FAKE, 64, None, 0, FAKE, 1e-5, FAKE, 64, None) == 1           # 64 % 24 != 0
    assert f(1, 4, 64, 0, FAKE, 64, None, 0, FAKE, -1.0, FAKE, 64, None) == 1            # eps < 0
    assert f(1, 4, 130, 1, FAKE, 130, None, 0, FAKE, 1e-5, FAKE, 130, None) == 2         # > 64 groups
    assert f(1, 4, 64, 0, FAKE + 2, 64, None, 0, FAKE, 1e-5, FAKE, 64, None) == 2        # misaligned


@pytest.mark.parametrize("lo,hi", [(-0.1, 1.0), (0.5, 0.1), (float("nan"), 1.0), (0.0, float("nan"))])
def test_bad_dt_limit_rejected_on_host(lib, lo, hi):
    d = pkg.Dims(1, 8, 2, 64, 1, 128)
    lim = pkg.DtLimit(lo, hi)
    assert lib.ssd_fwd_ex(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 1, FAKE, None,
                          ctypes.byref(lim), None, 0, None, 0, None) == 1
    d1 = pkg.Dims(1, 1, 2, 64, 1, 128)
    assert lib.ssd_step_ex(ctypes.byref(d1), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1, FAKE,
                           ctypes.byref(lim), None) == 1


def test_misaligned_seq_idx_is_unsupported(lib):
    d = pkg.Dims(1, 8, 2, 64, 1, 128)
    assert lib.ssd_fwd_ex(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 256, 1, FAKE, None,
                          None, FAKE + 2, 0, None, 0, None) == 2


def test_input_guard_rejects_bad_arguments_on_host(lib):
    d = pkg.Dims(1, 8, 2, 64, 1, 128)
    counts = (ctypes.c_int64 * 8)()
    f = lib.ssd_check_inputs
    assert f(None, 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 1    # no dims
    assert f(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None) == 1  # no counts
    assert f(ctypes.byref(d), 1, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 1  # no x
    assert f(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, counts, None) == 1  # no C
    assert f(ctypes.byref(d), 7, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 1  # dtype
    bad = pkg.Dims(1, 8, 3, 64, 2, 128)                                                           # 3 % 2
    assert f(ctypes.byref(bad), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 1
    # element alignment only: bf16 x may sit at 2 bytes, fp32 x or dt may not
    assert f(ctypes.byref(d), 1, FAKE + 1, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 2
    assert f(ctypes.byref(d), 0, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 2
    assert f(ctypes.byref(d), 1, FAKE, FAKE + 2, FAKE, FAKE, FAKE, FAKE, None, None, counts, None) == 2
    assert f(ctypes.byref(d), 1, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, None, counts, None) == 2


def test_host_entry_point_slice_rule(lib, monkeypatch):
    # one token slice per 96 MiB of copies (x and y in the io dtype, dt, B and C),
    # at least 4 and at most 16, none shorter than 512 tokens
    monkeypatch.delenv("SSD_HOST_SLICES", raising=False)
    f = pkg.ssd_host_slices
    assert f(4, 4096, 80, 64, 1, 128) == 4          # the 2.7B layer: 349 MB of copies
    assert f(1, 131072, 64, 64, 1, 256) == 16       # long context: 2.3 GB, capped
    assert f(2, 16000, 128, 64, 8, 128) == 12       # 1.2 GB
    assert f(8, 2048, 24, 64, 1, 128) == 4          # 111 MB: the minimum
    assert f(2, 1536, 4, 64, 2, 128) == 3           # 512-token floor
    assert f(2, 1023, 4, 64, 2, 128) == 1
    assert f(1, 1, 2, 64, 1, 128) == 1
    assert f(0, 4096, 80, 64, 1, 128) == 0          # invalid dims
    assert f(1, 4096, 6, 64, 4, 128) == 0
    monkeypatch.setenv("SSD_HOST_SLICES", "16")
    assert f(1, 8192, 2, 64, 1, 128) == 16
    assert f(2, 2600, 4, 64, 2, 128) == 5           # still no slice below 512 tokens
    monkeypatch.setenv("SSD_HOST_SLICES", "17")     # out of range: the rule from the copies
    assert f(4, 4096, 80, 64, 1, 128) == 4
