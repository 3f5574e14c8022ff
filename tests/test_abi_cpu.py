"""CPU-only checks of the C ABI: the library loads, exports every symbol that
include/samu.h declares, and rejects bad arguments on the host before any
CUDA call (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "samu.h")


@pytest.fixture(scope="module")
def lib():
    from linear_recurrence_sequence_gb300 import api
    if not os.path.exists(api.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return api._load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ["samu_forward", "samu_backward", "samu_workspace_bytes", "rglru_forward",
              "rglru_backward", "rglru_workspace_bytes", "lrs_status_string", "lrs_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from linear_recurrence_sequence_gb300 import api
    out = subprocess.run(["nm", "-D", "--defined-only", api.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert lib.lrs_status_string(0) == b"ok"
    for s in (1, 2, 3, 4):
        assert len(lib.lrs_status_string(s)) > 5
    assert lib.lrs_version() >= 100


def _ws(lib, fn, B, L, D):
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    st = getattr(lib, fn)(B, L, D, ctypes.byref(s), ctypes.byref(c))
    return st, s.value, c.value


def test_workspace_sizes(lib):
    st, saved, scratch = _ws(lib, "samu_workspace_bytes", 1, 32768, 2048)
    assert st == 0
    BL, M, S = 32768, 1024, 32768 // 16
    # controller cache (p, r, E-1/C/S/reset) + one entry state per 16-token sub-chunk at least
    assert saved >= BL * (4 + 4 + 16) + (S + 1) * M * 8
    assert saved % 256 == 0 and scratch % 256 == 0
    # bigger problems need at least as much workspace
    st2, saved2, scratch2 = _ws(lib, "samu_workspace_bytes", 2, 32768, 2048)
    assert saved2 > saved and scratch2 > scratch
    st, saved, scratch = _ws(lib, "rglru_workspace_bytes", 8, 16384, 1024)
    assert st == 0 and saved >= 8 * (16384 // 16 + 1) * 1024 * 4


@pytest.mark.parametrize("B,L,D,expect", [
    (0, 16, 64, 1), (1, 0, 64, 1), (1, 16, 63, 1), (1, 16, -2, 1),
    (1, 16, 12, 2), (1, 16, 8, 2), (1, 16, 24, 2), (1, 16, 4112, 2), (1, 16, 16, 0), (1, 1, 4096, 0),
])
def test_samu_shape_validation(lib, B, L, D, expect):
    st, _, _ = _ws(lib, "samu_workspace_bytes", B, L, D)
    assert st == expect


def test_rglru_width_rules(lib):
    assert _ws(lib, "rglru_workspace_bytes", 1, 5, 8)[0] == 0
    assert _ws(lib, "rglru_workspace_bytes", 1, 5, 1304)[0] == 0
    assert _ws(lib, "rglru_workspace_bytes", 1, 5, 6)[0] == 2
    assert _ws(lib, "rglru_workspace_bytes", 1, 5, 3)[0] == 1


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_forward_rejects_null_and_misaligned_pointers(lib):
    good = _fake(1 << 20)
    args = [good] * 10 + [1, 16, 64] + [good] * 5 + [None]
    # h0 = NULL and reset = NULL are allowed, the rest is checked; misaligned x_sel:
    bad = list(args)
    bad[0] = _fake((1 << 20) + 2)
    assert lib.samu_forward(*bad) == 1
    bad = list(args)
    bad[1] = None       # w is required
    assert lib.samu_forward(*bad) == 1
    bad = list(args)
    bad[13] = None      # y is required
    assert lib.samu_forward(*bad) == 1
    # odd width is an argument error even with valid pointers
    bad = list(args)
    bad[12] = 63
    assert lib.samu_forward(*bad) == 1


def test_backward_rejects_bad_grad_dtype(lib):
    good = _fake(1 << 20)
    args = [good] * 12 + [1, 16, 64] + [good, good, good, 7] + [good] * 8 + [None]
    assert lib.samu_backward(*args) == 1
    rg = [good] * 8 + [1, 16, 64] + [good] * 4 + [9] + [good] * 3 + [None]
    assert lib.rglru_backward(*rg) == 1


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from linear_recurrence_sequence_gb300 import api
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "_HERE", str(tmp_path))
    with pytest.raises(RuntimeError, match="not built"):
        api._load()


def test_chunk_transition_setting(lib):
    """Host-only: the process-wide item-transition form (closed form by default)."""
    assert lib.samu_get_chunk_transition() == 1
    assert lib.samu_set_chunk_transition(0) == 0
    assert lib.samu_get_chunk_transition() == 0
    assert lib.samu_set_chunk_transition(7) == 1          # LRS_ERR_ARG, setting unchanged
    assert lib.samu_get_chunk_transition() == 0
    assert lib.samu_set_chunk_transition(1) == 0
    assert lib.samu_get_chunk_transition() == 1


@pytest.mark.parametrize("B,L,D,expect", [
    (8, 8192, 1024, 0), (1, 200, 2048, 0), (1, 16, 1536, 0), (1, 16, 128, 0),
    (1, 16, 64, 2), (1, 16, 1000, 2), (1, 16, 1032, 2), (0, 16, 1024, 1),
])
def test_rglru_proj_shape_validation(lib, B, L, D, expect):
    """Host-only: the projected RG-LRU needs D a multiple of 128 (16 diagonal
    blocks whose width is a multiple of 8)."""
    st, saved, scratch = _ws(lib, "rglru_proj_workspace_bytes", B, L, D)
    assert st == expect
    if st == 0:
        # the FP32 logits of both gates and the six BF16 gradient parts per token at least
        assert scratch >= B * L * D * (8 + 12)
        st2, saved2, _ = _ws(lib, "rglru_workspace_bytes", B, L, D)
        assert st2 == 0 and saved == saved2


def test_projected_rglru_entry_points_reject_null_pointers(lib):
    """Host-only argument checks return LRS_ERR_ARG before any CUDA call."""
    null = ctypes.c_void_p(0)
    st = lib.rglru_proj_forward(null, null, null, null, null, null, null, null, 1, 16, 128,
                                null, null, null, null, null, null)
    assert st == 1
    st = lib.rglru_proj_backward(null, null, null, null, null, null, null, null, null, null, 1, 16, 128,
                                 null, null, 0, null, null, null, null, null, null, null, null)
    assert st == 1


def test_noalloc_size_limit_is_checked_before_any_device_call(lib):
    """samu_forward_noalloc refuses shapes whose intermediates exceed
    LRS_NOALLOC_BYTES before it touches the device.  Without a GPU, a shape
    that fits gets past that check and fails at the device look-up instead
    (LRS_ERR_CUDA); B=1, L=32768, D=2048 must fit, B=1, L=131072, D=1024 not."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: with a device the call would launch kernels")
    text = open(HEADER).read()
    assert re.search(r"#define LRS_NOALLOC_BYTES \(64u << 20\)", text)
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    LRS_ERR_CUDA, LRS_ERR_TOO_LARGE = 3, 5
    args = [p, p, None, None, p, p, p, p, p, p]
    assert lib.samu_forward_noalloc(*args, 1, 32768, 2048, p, None, p, None) == LRS_ERR_CUDA
    assert lib.samu_forward_noalloc(*args, 1, 32768, 2560, p, None, p, None) == LRS_ERR_CUDA
    assert lib.samu_forward_noalloc(*args, 1, 131072, 1024, p, None, p, None) == LRS_ERR_TOO_LARGE
    assert lib.samu_status_string(LRS_ERR_TOO_LARGE) == lib.lrs_status_string(LRS_ERR_TOO_LARGE)


def _block_ws(lib, B, L, Dm, D):
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    st = lib.samu_block_workspace_bytes(B, L, Dm, D, ctypes.byref(s), ctypes.byref(c))
    return st, s.value, c.value


@pytest.mark.parametrize("B,L,Dm,D,expect", [
    (4, 4096, 1024, 1024, 0), (1, 8192, 2048, 2560, 0), (2, 100, 256, 256, 0), (1, 16, 4096, 256, 0),
    (1, 16, 384, 256, 2), (1, 16, 256, 384, 2), (1, 16, 8192, 256, 2), (1, 16, 256, 4352, 2),
    (0, 16, 256, 256, 1), (1, 16, 0, 256, 1), (1, 16, 256, 255, 1),
])
def test_block_shape_validation(lib, B, L, Dm, D, expect):
    """Host-only: the block needs Dm and D multiples of 256 (the contraction
    tiles' 256 columns), Dm <= 4096 and D within the mixer's limits; its saved
    buffer holds the mixer's plus the BF16 activations of every layer."""
    st, saved, scratch = _block_ws(lib, B, L, Dm, D)
    assert st == expect
    if st == 0:
        mixer_saved = _ws(lib, "samu_workspace_bytes", B, L, D)[1]
        F = 3 * Dm
        # h1, r1, h2 (Dm each), [g|v] (2D), u, y, j (D each), [a|b] (2F), q (F): BF16
        assert saved >= mixer_saved + B * L * 2 * (3 * Dm + 5 * D + 3 * F)
        assert scratch > _ws(lib, "samu_workspace_bytes", B, L, D)[2]


def test_block_entry_points_reject_null_pointers(lib):
    """Host-only argument checks return LRS_ERR_ARG before any CUDA call."""
    null = ctypes.c_void_p(0)
    assert lib.samu_block_forward(null, null, null, null, 1, 16, 256, 256, null, null, null, null, null) == 1
    assert lib.samu_block_backward(null, null, null, null, null, null, 1, 16, 256, 256, null, null, null, null,
                                   null, null) == 1
    assert lib.lrs_dense_gemm(0, null, null, null, 128, 256, 64, null, null) == 1
    buf = (ctypes.c_uint8 * 4096)()
    p = ctypes.c_void_p((ctypes.addressof(buf) + 255) // 256 * 256)
    assert lib.lrs_dense_gemm(3, p, p, p, 128, 256, 64, p, null) == 1          # unknown layout
    assert lib.lrs_dense_gemm(0, p, p, p, 128, 192, 64, p, null) == 2          # N not a multiple of 256
    assert lib.lrs_dense_gemm(2, p, p, p, 100, 256, 64, p, null) == 2          # TN: M not a multiple of 128


@pytest.mark.parametrize("B,L,Dm,D,expect", [
    (4, 4096, 1024, 1024, 0), (1, 8192, 2048, 2560, 0), (2, 100, 256, 256, 0), (1, 16, 256, 8192, 0),
    (1, 16, 384, 256, 2), (1, 16, 256, 384, 2), (0, 16, 256, 256, 1), (1, 16, 0, 256, 1),
])
def test_rglru_block_shape_validation(lib, B, L, Dm, D, expect):
    """Host-only: the RG-LRU block follows the block's width rules and the
    projected RG-LRU's (no SAMU width limit: D = 8192 is accepted)."""
    s = ctypes.c_size_t(0)
    c = ctypes.c_size_t(0)
    st = lib.rglru_block_workspace_bytes(B, L, Dm, D, ctypes.byref(s), ctypes.byref(c))
    assert st == expect
    if st == 0:
        st2, msaved, _ = _ws(lib, "rglru_proj_workspace_bytes", B, L, D)
        assert st2 == 0 and s.value >= msaved + B * L * 2 * (3 * Dm + 5 * D + 9 * Dm)


def test_rglru_block_entry_points_reject_null_pointers(lib):
    null = ctypes.c_void_p(0)
    assert lib.rglru_block_forward(null, null, null, null, 1, 16, 256, 256, null, null, null, null, null) == 1
    assert lib.rglru_block_backward(null, null, null, null, null, null, 1, 16, 256, 256, null, null, null, null,
                                    null, null) == 1
