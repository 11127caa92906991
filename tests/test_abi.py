"""The C-ABI library: it builds, loads, exports every symbol include/fa2.h declares,
and rejects invalid arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re
import threading

import pytest

from attention_fa2_forward_02_gb300 import binding
from attention_fa2_forward_02_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA_ERR, TIMEOUT, WORKSPACE = range(7)
F32, F16, BF16 = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return binding.library()


def declared_functions():
    names = []
    for fname in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_calls():
    names = declared_functions()
    for n in ("fa2_forward", "fa2_backward", "fa2_backward_workspace_size", "psa_pack_qkv", "psa_merge_attn_nchw",
              "fa2_status_string", "fa2_device_status"):
        assert n in names
    assert set(binding.EXPORTS) <= set(names)


def test_binding_rejects_a_tensor_of_another_device(monkeypatch):
    """The binding refuses, before any library call, a tensor that is not on the current
    device (the kernels would run on the current one). A stand-in tensor and a patched
    current device: no GPU needed."""
    torch = pytest.importorskip("torch")

    class FakeCudaTensor:
        is_cuda = True
        device = torch.device("cuda", 1)

        def is_contiguous(self):
            return True

        def dim(self):
            return 3

        def data_ptr(self):
            return 0

    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    with pytest.raises(ValueError, match="current device"):
        binding._dev(FakeCudaTensor(), "q", 3)
    FakeCudaTensor.device = torch.device("cuda", 0)
    assert binding._dev(FakeCudaTensor(), "q", 3).value is None  # accepted: a null pointer's c_void_p


def test_launch_record_of_a_thread_that_launched_nothing(lib):
    """fa2_last_launch_info: all zero on a host thread that has launched nothing; a call that
    fails validation leaves the record alone; NULL is an invalid argument. No GPU needed."""
    out = {}

    def run():
        info = binding.LaunchInfo()
        # a forward with null pointers: rejected before any launch or record
        out["fwd"] = lib.fa2_forward(None, None, None, None, None, 1, 1, 1, 64, BF16, 0.125, None)
        out["st"] = lib.fa2_last_launch_info(ctypes.byref(info))
        out["info"] = [getattr(info, f) for f, _ in binding.LaunchInfo._fields_]
        out["null"] = lib.fa2_last_launch_info(None)

    t = threading.Thread(target=run)
    t.start()
    t.join()
    assert out["fwd"] == 1  # FA2_ERR_INVALID_ARG
    assert out["st"] == 0 and out["info"] == [0, 0, 0, 0, 0]
    assert out["null"] == 1


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(8):
        msg = lib.fa2_status_string(s).decode()
        assert msg and msg != "unknown status"
    assert lib.fa2_status_string(99).decode() == "unknown status"


P = ctypes.c_void_p(0x1000)        # never dereferenced: every call below fails validation first
PM = ctypes.c_void_p(0x1008)       # misaligned


def fwd(lib, q=P, k=P, v=P, o=P, l=P, bh=2, nq=64, nk=64, d=64, dt=BF16, scale=0.125):
    return lib.fa2_forward(q, k, v, o, l, bh, nq, nk, d, dt, scale, None)


@pytest.mark.parametrize("kw,want", [
    ({"q": None}, INVALID), ({"l": None}, INVALID), ({"bh": 0}, INVALID), ({"nq": 0}, INVALID), ({"nk": -1}, INVALID),
    ({"d": 0}, INVALID), ({"dt": 7}, INVALID), ({"scale": 0.0}, INVALID), ({"scale": float("nan")}, INVALID),
    ({"scale": float("inf")}, INVALID), ({"d": 12}, UNSUPPORTED), ({"d": 136}, UNSUPPORTED), ({"d": 7}, UNSUPPORTED),
    ({"d": 129, "dt": F32}, UNSUPPORTED), ({"d": 12, "dt": F16}, UNSUPPORTED),
    ({"bh": 70000}, UNSUPPORTED), ({"q": PM}, MISALIGNED), ({"o": PM}, MISALIGNED),
])
def test_forward_validation(lib, kw, want):
    assert fwd(lib, **kw) == want


def test_backward_validation(lib):
    args = [P] * 9
    assert lib.fa2_backward(*args, P, 1 << 20, 2, 64, 64, 64, F32, 0.125, None) == UNSUPPORTED
    assert lib.fa2_backward(*args, None, 1 << 20, 2, 64, 64, 64, BF16, 0.125, None) == WORKSPACE
    assert lib.fa2_backward(*args, P, 16, 2, 64, 64, 64, BF16, 0.125, None) == WORKSPACE
    assert lib.fa2_backward(*args, PM, 1 << 20, 2, 64, 64, 64, BF16, 0.125, None) == WORKSPACE
    assert lib.fa2_backward(None, *args[1:], P, 1 << 20, 2, 64, 64, 64, BF16, 0.125, None) == INVALID
    assert lib.fa2_backward(*args, P, 1 << 20, 2, 64, 64, 44, BF16, 0.125, None) == UNSUPPORTED
    assert lib.fa2_backward(*args[:6], PM, *args[7:], P, 1 << 20, 2, 64, 64, 64, BF16, 0.125, None) == MISALIGNED


def test_workspace_size(lib):
    assert lib.fa2_backward_workspace_size(2, 100, 50, 64, BF16) >= 2 * 100 * 4
    assert lib.fa2_backward_workspace_size(0, 100, 50, 64, BF16) == 0
    assert lib.fa2_backward_workspace_size(2, 100, 50, 44, BF16) == 0
    assert lib.fa2_backward_workspace_size(2, 100, 50, 48, BF16) >= 2 * 100 * 4


def test_psa_validation(lib):
    # qkv_h not a multiple of 4*num_heads
    assert lib.psa_pack_qkv(P, P, 100, 20, 20, 8, 4, F16, None) == INVALID
    assert lib.psa_pack_qkv(None, P, 512, 20, 20, 8, 4, F16, None) == INVALID
    assert lib.psa_pack_qkv(P, P, 512, 0, 20, 8, 4, F16, None) == INVALID
    assert lib.psa_pack_qkv(P, P, 512, 20, 20, 8, 4, 9, None) == INVALID
    assert lib.psa_pack_qkv(PM, P, 512, 20, 20, 8, 4, F16, None) == MISALIGNED
    assert lib.psa_merge_attn_nchw(P, P, P, 250, 20, 20, 8, 4, F16, None) == INVALID
    assert lib.psa_merge_attn_nchw(P, None, P, 256, 20, 20, 8, 4, F16, None) == INVALID
    assert lib.psa_merge_attn_nchw(P, P, PM, 256, 20, 20, 8, 4, F16, None) == MISALIGNED


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(binding.Fa2Error):
        saved = binding._lib
        try:
            binding._lib = None
            binding.library(str(tmp_path / "missing.so"))
        finally:
            binding._lib = saved


def test_binding_rejects_mixed_dtypes(lib):
    """Every wrapper that hands the library one dtype code for several tensors checks that
    they share that dtype (the library would otherwise read one type as another)."""
    torch = pytest.importorskip("torch")
    bh, n, d = 1, 16, 32
    bf = lambda *s: torch.zeros(s, dtype=torch.bfloat16)  # noqa: E731
    hf = lambda *s: torch.zeros(s, dtype=torch.float16)  # noqa: E731
    f32 = lambda *s: torch.zeros(s, dtype=torch.float32)  # noqa: E731
    q, k, v, o, do = (bf(bh, n, d) for _ in range(5))
    lse, ws = f32(bh, n), torch.zeros(4096, dtype=torch.uint8)
    odd = hf(bh, n, d)
    with pytest.raises(TypeError):
        binding.fa2_backward(q, k, v, o, do, lse, odd, bf(bh, n, d), bf(bh, n, d), ws, 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward(q, k, odd, o, do, lse, bf(bh, n, d), bf(bh, n, d), bf(bh, n, d), ws, 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward(q, k, v, o, do, f32(bh, n).half(), bf(bh, n, d), bf(bh, n, d), bf(bh, n, d), ws, 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward_noalloc(q, k, v, odd, do, lse, bf(bh, n, d), bf(bh, n, d), bf(bh, n, d), 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward_preprocess(o, odd, lse, ws, n)
    with pytest.raises(TypeError):
        binding.fa2_backward_dkdv(q, k, v, do, ws, odd, bf(bh, n, d), 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward_dq(q, k, v, odd, ws, bf(bh, n, d), 0.17)
    with pytest.raises(TypeError):
        binding.fa2_backward_passes(q, k, v, do, ws, bf(bh, n, d), bf(bh, n, d), odd, 0.17)
    packed = bf(4, bh, n, d)
    with pytest.raises(TypeError):
        binding.psa_fa2_forward(packed, bf(bh, n, d), odd, lse, 0.17)
    with pytest.raises(TypeError):
        binding.psa_fa2_backward(packed, o, o, do, odd, lse, bf(4, bh, n, d), ws, 0.17)
    with pytest.raises(TypeError):
        binding.psa_merge_attn_backward(bf(1, 2 * d, 4, 4), hf(1, 16, d), bf(1, 16, d), 1)


def test_workspace_holds_the_split_dq_partial_sums(lib):
    """Head size > 64: the workspace adds room for the split dQ pass's float32 partial sums
    exactly when the unsplit dQ CTAs would be fewer than about 148 (fa2.h)."""
    ws = lambda bh, nq, nk, d: lib.fa2_backward_workspace_size(bh, nq, nk, d, BF16)  # noqa: E731
    pad = lambda n: -(-n // 128) * 128  # noqa: E731
    # 2 heads x 1 query tile, 256 key tiles: 8 ranges
    assert ws(2, 128, 32768, 128) == 8 * 2 * 128 + 8 * 2 * 128 * 128 * 4
    # 1 head x 3 query tiles, 64 key tiles: 8 ranges; head size 120 runs at 128
    assert ws(1, 300, 8192, 120) == 8 * pad(300) + 8 * 1 * pad(300) * 128 * 4
    # 3 heads x 2 query tiles, 20 key tiles: min(ceil(148 / 6), 20 // 8) = 2 ranges
    assert ws(3, 200, 2500, 128) == 8 * 3 * pad(200) + 2 * 3 * pad(200) * 128 * 4
    # a wave of dQ CTAs or more (B=1 H=32 N_q=1024: 256), or fewer than 16 key tiles: no split
    assert ws(32, 1024, 32768, 128) == 8 * 32 * 1024
    assert ws(32, 8192, 8192, 128) == 8 * 32 * 8192
    assert ws(2, 128, 1900, 128) == 8 * 2 * 128
    # head size <= 64: the one-pass workspace (D, LSE2 and the dQ accumulator)
    assert ws(2, 128, 32768, 64) == 8 * 2 * 128 + 2 * 128 * 64 * 4
