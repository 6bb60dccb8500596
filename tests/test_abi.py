"""Host-side checks of the C ABI: the library loads, exports every function
that include/kda.h declares, and rejects bad arguments before any launch
(no device memory is touched: every pointer here is NULL or a host array)."""
import ctypes
import os
import re

import pytest

import kimi_delta_attention_rule_gb300 as kda
from kimi_delta_attention_rule_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    import glob
    src = "".join(open(p).read() for p in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 7
    for name in names:
        assert hasattr(lib, name), name
    assert set(kda.EXPORTED) <= set(names)


def test_status_strings(lib):
    for code, name in [(0, "KDA_OK"), (1, "KDA_ERR_INVALID_ARG"), (2, "KDA_ERR_UNSUPPORTED"),
                       (3, "KDA_ERR_CUDA"), (4, "KDA_ERR_TIMEOUT"), (5, "KDA_ERR_DEVICE"),
                       (6, "KDA_ERR_TOO_LARGE"), (7, "KDA_ERR_RANGE")]:
        assert kda.status_string(code) == name
    assert kda.status_string(99) == "KDA_ERR_UNKNOWN"
    assert lib.kda_abi_version() == 101


def test_workspace_size(lib):
    # bf16: status word + one prepared block (BLOCK bytes) and one 4-byte ready
    # flag per (chunk, head)
    BLOCK = 74368
    assert kda.kda_prefill_workspace_size(1, 8192, 32, 128, 64, kda.KDA_BF16) >= 128 * 32 * BLOCK
    assert kda.kda_prefill_workspace_size(4, 100, 2, 128, 64, kda.KDA_BF16) >= 4 * 2 * 2 * BLOCK
    # packed: T is the total; one spare chunk slot per sequence at most
    vl = kda.kda_prefill_workspace_size(64, 1 << 20, 32, 128, 64, kda.KDA_BF16, varlen=True)
    assert ((1 << 20) // 64) * 32 * BLOCK <= vl <= ((1 << 20) // 64 + 64) * 32 * (BLOCK + 4) + 4096
    assert kda.kda_prefill_workspace_size(1, 64, 2, 128, 16, kda.KDA_F32) >= 256
    assert kda.kda_prefill_workspace_size(1, 64, 2, 64, 64, kda.KDA_BF16) == 0      # D != 128
    assert kda.kda_prefill_workspace_size(1, 64, 2, 128, 16, kda.KDA_BF16) == 0     # chunk
    assert kda.kda_prefill_workspace_size(-1, 64, 2, 128, 64, kda.KDA_BF16) == 0


def _prefill(lib, **kw):
    a = dict(q=None, k=None, v=None, g=None, beta=None, scale=1.0, init=None, cu=None, N=1, T=64,
             H=2, D=128, chunk=64, io=0, out=None, fin=None, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.kda_prefill(a["q"], a["k"], a["v"], a["g"], a["beta"], a["scale"], a["init"],
                           a["cu"], a["N"], a["T"], a["H"], a["D"], a["chunk"], a["io"], a["out"],
                           a["fin"], a["ws"], a["ws_bytes"], a["stream"])


def test_prefill_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    assert _prefill(lib, D=64) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, chunk=32) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, io=7) == kda.KDA_ERR_UNSUPPORTED
    assert _prefill(lib, N=-1) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib, H=0) == kda.KDA_ERR_INVALID_ARG
    assert _prefill(lib) == kda.KDA_ERR_INVALID_ARG                      # no workspace
    assert _prefill(lib, ws=fake, ws_bytes=16) == kda.KDA_ERR_INVALID_ARG  # too small
    assert _prefill(lib, ws=ctypes.c_void_p(0x100010), ws_bytes=256) == kda.KDA_ERR_INVALID_ARG
    big = 1 << 40
    assert _prefill(lib, ws=fake, ws_bytes=256) == kda.KDA_ERR_INVALID_ARG  # workspace too small
    assert _prefill(lib, ws=fake, ws_bytes=big) == kda.KDA_ERR_INVALID_ARG  # null tensors
    mis = ctypes.c_void_p(0x100002)
    assert _prefill(lib, q=mis, k=fake, v=fake, g=fake, beta=fake, out=fake, ws=fake,
                    ws_bytes=big) == kda.KDA_ERR_INVALID_ARG             # misaligned q
    assert _prefill(lib, N=1, T=1 << 31 - 1, H=1 << 12, ws=fake, ws_bytes=256) \
        == kda.KDA_ERR_INVALID_ARG                                       # size overflow
    # N = 0 is a valid empty call: nothing is launched
    assert _prefill(lib, N=0, ws=fake, ws_bytes=256) == kda.KDA_OK


def test_prefill_schedule_query(lib):
    f = lib.kda_prefill_schedule
    # invalid sizes: the negated status, no device needed
    assert f(1, 64, 2, 64, 64, kda.KDA_BF16, 0) == -kda.KDA_ERR_UNSUPPORTED
    assert f(1, 64, 2, 128, 16, kda.KDA_BF16, 0) == -kda.KDA_ERR_UNSUPPORTED
    assert f(-1, 64, 2, 128, 64, kda.KDA_BF16, 0) == -kda.KDA_ERR_INVALID_ARG
    # fp32 I/O has one schedule
    assert f(1, 64, 2, 128, 16, kda.KDA_F32, 0) == kda.KDA_SCHEDULE_DIRECT
    assert kda.kda_prefill_schedule(3, 100, 2, 128, 64, kda.KDA_F32, True) == \
        kda.KDA_SCHEDULE_DIRECT
    with pytest.raises(kda.KDAError):
        kda.kda_prefill_schedule(1, 64, 0, 128, 64, kda.KDA_BF16)


def test_decode_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    f = lib.kda_decode_step
    assert f(None, None, None, None, None, 1.0, 4, 2, 64, 0, None, None, None) == kda.KDA_ERR_UNSUPPORTED
    assert f(None, None, None, None, None, 1.0, 4, 2, 128, 3, None, None, None) == kda.KDA_ERR_UNSUPPORTED
    assert f(None, None, None, None, None, 1.0, -1, 2, 128, 0, None, None, None) == kda.KDA_ERR_INVALID_ARG
    assert f(None, None, None, None, None, 1.0, 4, 2, 128, 0, None, None, None) == kda.KDA_ERR_INVALID_ARG
    assert f(fake, fake, fake, fake, fake, 1.0, 4, 2, 128, 0, ctypes.c_void_p(0x100004), fake,
             None) == kda.KDA_ERR_INVALID_ARG                            # misaligned state
    assert f(None, None, None, None, None, 1.0, 0, 2, 128, 0, None, None, None) == kda.KDA_OK


def test_prefill_ex_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    f = lib.kda_prefill_ex
    def call(gpc=1, si=0, smax=0, snaps=None, chunk=64, ws_bytes=1 << 40):
        return f(fake, fake, fake, fake, fake, 1.0, None, None, 1, 128, 2, 128, chunk, 0, gpc, si,
                 smax, snaps, fake, None, fake, ws_bytes, None)
    assert call(gpc=2) == kda.KDA_ERR_INVALID_ARG
    assert call(si=-64) == kda.KDA_ERR_INVALID_ARG
    assert call(si=96, smax=2, snaps=fake) == kda.KDA_ERR_UNSUPPORTED   # not a multiple of 64
    assert call(si=64, smax=2, snaps=None) == kda.KDA_ERR_INVALID_ARG   # nowhere to write
    assert call(si=64, smax=0, snaps=fake) == kda.KDA_ERR_INVALID_ARG
    assert call(si=64, smax=2, snaps=ctypes.c_void_p(0x100008)) == kda.KDA_ERR_INVALID_ARG
    assert call(ws_bytes=16) == kda.KDA_ERR_INVALID_ARG                  # workspace too small


def test_decode_multi_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    f = lib.kda_decode
    args = lambda **kw: dict(dict(q=fake, k=fake, v=fake, g=fake, beta=fake, B=4, T=2, H=2, D=128,
                                  io=0, gpc=1, pool=fake, P=4, idx=None, out=fake), **kw)
    call = lambda a: f(a["q"], a["k"], a["v"], a["g"], a["beta"], 1.0, a["B"], a["T"], a["H"],
                       a["D"], a["io"], a["gpc"], a["pool"], a["P"], a["idx"], a["out"], None)
    assert call(args(T=65)) == kda.KDA_ERR_UNSUPPORTED        # beyond a chunk
    assert call(args(D=64)) == kda.KDA_ERR_UNSUPPORTED
    assert call(args(io=5)) == kda.KDA_ERR_UNSUPPORTED
    assert call(args(gpc=2)) == kda.KDA_ERR_INVALID_ARG
    assert call(args(P=3)) == kda.KDA_ERR_INVALID_ARG         # pool smaller than B, no indices
    assert call(args(T=-1)) == kda.KDA_ERR_INVALID_ARG
    assert call(args(pool=ctypes.c_void_p(0x100004))) == kda.KDA_ERR_INVALID_ARG  # misaligned
    mis = ctypes.c_void_p(0x100008)  # input rows are copied in 16-byte pieces
    for name in ("q", "k", "v", "g", "out"):
        assert call(args(**{name: mis})) == kda.KDA_ERR_INVALID_ARG, name
    # a scalar decay per (token, head) is read element by element: any alignment
    assert call(args(g=mis, gpc=0, B=0)) == kda.KDA_OK
    assert call(args(q=None)) == kda.KDA_ERR_INVALID_ARG
    assert call(args(B=0)) == kda.KDA_OK and call(args(T=0)) == kda.KDA_OK  # nothing to do


def test_host_cu_seqlens_check(lib):
    assert kda.kda_check_cu_seqlens([0, 5, 5, 9], 9) == kda.KDA_OK
    assert kda.kda_check_cu_seqlens([0, 5, 3, 9], 9) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_check_cu_seqlens([1, 5, 9], 9) == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_check_cu_seqlens([0, 5, 8], 9) == kda.KDA_ERR_INVALID_ARG


def test_product_path_has_no_cpu_fallback():
    """The binding never imports the oracle and raises without the library."""
    import kimi_delta_attention_rule_gb300 as pkg
    src = open(pkg.__file__).read()
    assert "oracle" not in src.replace("no CPU fallback", "")
    for f in os.listdir(os.path.join(ROOT, "kimi_delta_attention_rule_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "kimi_delta_attention_rule_gb300", "csrc", f)).read()


def test_layer_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    odd = ctypes.c_void_p(0x100008)  # 8-byte aligned, not 16
    pro = lib.kda_layer_prologue
    def call_pro(W=4, D=128, io=0, T=16, H=2, conv=fake, q=fake, g=fake):
        return pro(q, fake, fake, fake, fake, conv, fake, fake, W, None, 1, T, H, D, io, fake,
                   fake, fake, g, fake, None)
    assert call_pro(W=0) == kda.KDA_ERR_UNSUPPORTED and call_pro(W=5) == kda.KDA_ERR_UNSUPPORTED
    assert call_pro(D=64) == kda.KDA_ERR_UNSUPPORTED and call_pro(io=7) == kda.KDA_ERR_UNSUPPORTED
    assert call_pro(T=-1) == kda.KDA_ERR_INVALID_ARG and call_pro(H=0) == kda.KDA_ERR_INVALID_ARG
    assert call_pro(q=None) == kda.KDA_ERR_INVALID_ARG
    assert call_pro(q=ctypes.c_void_p(0x100004)) == kda.KDA_ERR_INVALID_ARG  # bf16 rows: 8 B
    assert call_pro(io=1, q=odd) == kda.KDA_ERR_INVALID_ARG                  # fp32 rows: 16 B
    assert call_pro(g=odd) == kda.KDA_ERR_INVALID_ARG
    assert call_pro(conv=odd) == kda.KDA_ERR_INVALID_ARG                     # weights: 16 B
    assert call_pro(T=0) == kda.KDA_OK
    epi = lib.kda_layer_epilogue
    def call_epi(D=128, io=0, T=16, o=fake, w=fake):
        return epi(o, fake, w, T, 2, D, io, fake, None)
    assert call_epi(D=64) == kda.KDA_ERR_UNSUPPORTED and call_epi(io=7) == kda.KDA_ERR_UNSUPPORTED
    assert call_epi(T=-1) == kda.KDA_ERR_INVALID_ARG and call_epi(o=None) == kda.KDA_ERR_INVALID_ARG
    assert call_epi(w=odd) == kda.KDA_ERR_INVALID_ARG
    assert call_epi(io=1, o=odd) == kda.KDA_ERR_INVALID_ARG
    assert call_epi(io=0, o=odd) == kda.KDA_ERR_INVALID_ARG  # bf16 rows too: 16 B per lane
    assert call_epi(T=0) == kda.KDA_OK


def test_schedule_override_validates_and_returns_the_previous_value(lib):
    # a process-wide setting: no device is touched
    assert lib.kda_prefill_set_schedule(7) == -kda.KDA_ERR_INVALID_ARG
    prev = kda.kda_prefill_set_schedule(kda.KDA_SCHEDULE_SPLIT)
    assert kda.kda_prefill_set_schedule(kda.KDA_SCHEDULE_FUSED) == kda.KDA_SCHEDULE_SPLIT
    assert kda.kda_prefill_set_schedule(prev) == kda.KDA_SCHEDULE_FUSED


def test_testing_entry_point_rejects_bad_arguments(lib):
    f = lib.kda_testing_prefill_chain_timeout
    args = [None] * 5 + [1.0, None, None, 1, 64, 2, 128, 64]
    assert f(*args, kda.KDA_F32, None, None, None, 0, 50, None) == kda.KDA_ERR_UNSUPPORTED
    assert f(*args, kda.KDA_BF16, None, None, None, 0, 0, None) == kda.KDA_ERR_INVALID_ARG
    assert f(*args, kda.KDA_BF16, None, None, None, 0, 50, None) == kda.KDA_ERR_INVALID_ARG


def test_layer_prologue_decode_argument_validation(lib):
    fake = ctypes.c_void_p(0x100000)
    f = lib.kda_layer_prologue_decode
    args = lambda **kw: dict(dict(W=4, B=2, T=1, H=2, D=128, io=0, st=fake, P=2, idx=None,
                                  p=fake), **kw)
    call = lambda a: f(a["p"], fake, fake, fake, fake, fake, fake, fake, a["W"], a["B"], a["T"],
                       a["H"], a["D"], a["io"], a["st"], a["P"], a["idx"], fake, fake, fake, fake,
                       fake, None)
    assert call(args(W=5)) == kda.KDA_ERR_UNSUPPORTED
    assert call(args(D=64)) == kda.KDA_ERR_UNSUPPORTED
    assert call(args(io=3)) == kda.KDA_ERR_UNSUPPORTED
    assert call(args(P=1)) == kda.KDA_ERR_INVALID_ARG           # pool smaller than B, no indices
    assert call(args(st=None)) == kda.KDA_ERR_INVALID_ARG       # W > 1 needs the state
    assert call(args(st=ctypes.c_void_p(0x100002))) == kda.KDA_ERR_INVALID_ARG  # misaligned
    assert call(args(p=ctypes.c_void_p(0x100004))) == kda.KDA_ERR_INVALID_ARG
    assert call(args(B=0)) == kda.KDA_OK and call(args(T=0)) == kda.KDA_OK
