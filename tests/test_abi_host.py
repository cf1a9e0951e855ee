"""Host-side checks of the C ABI: the library loads, exports every function
include/ssscan.h declares, and rejects bad arguments before touching a GPU.
No compute call is made here (this runs without a GPU)."""
import ctypes
import os
import re

import pytest

from selective_state_space_146_b300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssscan.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        from selective_state_space_146_b300.csrc import build
        build.build()
    return _abi.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ss_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared_functions()
    assert "ss_selective_scan_fwd" in names and "ss_ssd_chunk_scan_fwd" in names
    assert set(names) == set(_abi.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(0, -10, -1):
        s = _abi.status_string(code)
        assert s and s != "unknown status"
    assert _abi.status_string(-99) == "unknown status"
    assert lib.ss_version() >= 100


class FakeT:
    """Shape/stride/dtype description with a fake, aligned device address."""

    addr = 0x10000

    def __init__(self, shape, dtype=_abi.SS_BF16, stride=None, data=None):
        self.s = _abi.SSTensor()
        FakeT.addr += 0x100000
        self.s.data = FakeT.addr if data is None else data
        self.s.dtype = dtype
        self.s.ndim = len(shape)
        st = stride or [int(__import__("numpy").prod(shape[i + 1:])) for i in range(len(shape))]
        for i, (n, k) in enumerate(zip(shape, st)):
            self.s.shape[i] = n
            self.s.stride[i] = k

    @property
    def ref(self):
        return ctypes.byref(self.s)


def _sel_args(Bsz=2, D=8, N=16, L=64, dt=_abi.SS_BF16):
    u = FakeT((Bsz, D, L), dt)
    return dict(u=u, delta=FakeT((Bsz, D, L), dt), A=FakeT((D, N), _abi.SS_F32),
                B=FakeT((Bsz, N, L), dt), C=FakeT((Bsz, N, L), dt), D=FakeT((D,), _abi.SS_F32),
                z=FakeT((Bsz, D, L), dt), bias=FakeT((D,), _abi.SS_F32), y=FakeT((Bsz, D, L), dt),
                last=FakeT((Bsz, D, N), _abi.SS_F32))


def _call_sel(lib, a, softplus=1, drop=()):
    r = {k: (None if k in drop else v.ref) for k, v in a.items()}
    return lib.ss_selective_scan_fwd(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"], r["z"],
                                     r["bias"], softplus, r["y"], r["last"], None)


def test_selective_argument_errors(lib):
    a = _sel_args()
    assert _call_sel(lib, a, drop=("u",)) == -1
    assert _call_sel(lib, a, drop=("y",)) == -1
    assert _call_sel(lib, a, softplus=2) == -1
    b = _sel_args()
    b["delta"] = FakeT((2, 8, 63))
    assert _call_sel(lib, b) == -2
    b = _sel_args()
    b["B"] = FakeT((2, 15, 64))
    assert _call_sel(lib, b) == -2
    b = _sel_args()
    b["last"] = FakeT((2, 8, 8), _abi.SS_F32)
    assert _call_sel(lib, b) == -2
    b = _sel_args()
    b["z"] = FakeT((2, 8, 64), _abi.SS_F32)
    assert _call_sel(lib, b) == -3
    b = _sel_args()
    b["A"] = FakeT((8, 16), _abi.SS_BF16)
    assert _call_sel(lib, b) == -3
    b = _sel_args()
    b["u"] = FakeT((2, 8, 64), 7)
    assert _call_sel(lib, b) == -3
    b = _sel_args()
    b["u"] = FakeT((2, 8, 64), data=0x10001)  # odd address for a 2-byte element
    assert _call_sel(lib, b) == -4
    b = _sel_args(N=300)
    assert _call_sel(lib, b) == -5
    b = _sel_args()
    b["u"] = FakeT((2, 8, 64), stride=[512, 64, -1])
    assert _call_sel(lib, b) == -2


def test_selective_zero_size_is_a_no_op(lib):
    for shp in ((0, 8, 64), (2, 0, 64)):
        Bsz, D, L = shp
        a = _sel_args(Bsz, D, 16, L)
        assert _call_sel(lib, a) == 0
    a = _sel_args(2, 8, 16, 0)
    assert _call_sel(lib, a, drop=("last",)) == 0


def _ssd_args(Bsz=2, L=64, H=4, P=8, G=1, N=16, dt=_abi.SS_BF16):
    return dict(x=FakeT((Bsz, L, H, P), dt), dt=FakeT((Bsz, L, H), dt),
                A=FakeT((H,), _abi.SS_F32), B=FakeT((Bsz, L, G, N), dt),
                C=FakeT((Bsz, L, G, N), dt), D=FakeT((H,), _abi.SS_F32),
                y=FakeT((Bsz, L, H, P), dt), last=FakeT((Bsz, H, P, N), _abi.SS_F32))


def _call_ssd(lib, a, chunk=64, drop=()):
    r = {k: (None if k in drop else v.ref) for k, v in a.items()}
    return lib.ss_ssd_chunk_scan_fwd(r["x"], r["dt"], r["A"], r["B"], r["C"], r["D"], chunk,
                                     r["y"], r["last"], None)


def test_ssd_argument_errors(lib):
    assert _call_ssd(lib, _ssd_args(), chunk=100) == -1
    assert _call_ssd(lib, _ssd_args(), drop=("x",)) == -1
    a = _ssd_args(H=4, G=3)
    assert _call_ssd(lib, a) == -2
    a = _ssd_args()
    a["dt"] = FakeT((2, 64, 5))
    assert _call_ssd(lib, a) == -2
    a = _ssd_args()
    a["B"] = FakeT((2, 64, 1, 16), _abi.SS_F32)
    assert _call_ssd(lib, a) == -3
    a = _ssd_args(N=512)
    assert _call_ssd(lib, a) == -5
    a = _ssd_args(Bsz=0)
    assert _call_ssd(lib, a) == 0


def test_initial_state_and_step_argument_errors(lib):
    a = _sel_args()
    bad_h0 = FakeT((2, 8, 15), _abi.SS_F32)
    r = {k: v.ref for k, v in a.items()}
    assert lib.ss_selective_scan_fwd_init(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 1, bad_h0.ref, r["y"], r["last"],
                                          None) == -2
    bf_h0 = FakeT((2, 8, 16), _abi.SS_BF16)
    assert lib.ss_selective_scan_fwd_init(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 1, bf_h0.ref, r["y"], r["last"],
                                          None) == -3
    # one decode step: (batch, d_inner) activations, (batch, N) B / C
    st = FakeT((2, 8, 16), _abi.SS_F32)
    u, dl, z, y = (FakeT((2, 8)) for _ in range(4))
    Bm, Cm = FakeT((2, 16)), FakeT((2, 16))
    A, D, bias = FakeT((8, 16), _abi.SS_F32), FakeT((8,), _abi.SS_F32), FakeT((8,), _abi.SS_F32)
    assert lib.ss_selective_state_update(FakeT((2, 8, 8), _abi.SS_F32).ref, u.ref, dl.ref, A.ref,
                                         Bm.ref, Cm.ref, D.ref, z.ref, bias.ref, 1, y.ref,
                                         None) == -2
    assert lib.ss_selective_state_update(FakeT((2, 8, 16), _abi.SS_BF16).ref, u.ref, dl.ref,
                                         A.ref, Bm.ref, Cm.ref, D.ref, z.ref, bias.ref, 1, y.ref,
                                         None) == -3
    assert lib.ss_selective_state_update(st.ref, u.ref, dl.ref, A.ref, Bm.ref, Cm.ref, D.ref,
                                         z.ref, bias.ref, 5, y.ref, None) == -1
    # SSD step: groups must divide heads
    sst = FakeT((2, 4, 8, 16), _abi.SS_F32)
    x, yy = FakeT((2, 4, 8)), FakeT((2, 4, 8))
    dt = FakeT((2, 4))
    Ah, Dh = FakeT((4,), _abi.SS_F32), FakeT((4,), _abi.SS_F32)
    Bg, Cg = FakeT((2, 3, 16)), FakeT((2, 3, 16))
    assert lib.ss_ssd_state_update(sst.ref, x.ref, dt.ref, Ah.ref, Bg.ref, Cg.ref, Dh.ref, yy.ref,
                                   None) == -2


def _call_bwd(lib, a, g, softplus=1):
    r = {k: (None if v is None else v.ref) for k, v in a.items()}
    o = {k: (None if v is None else v.ref) for k, v in g.items()}
    return lib.ss_selective_scan_bwd(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"], r["z"],
                                     r["bias"], softplus, r["y"], o["du"], o["ddelta"], o["dA"],
                                     o["dB"], o["dC"], o["dD"], o["dz"], o["dbias"], None)


def _bwd_grads(Bsz=2, D=8, N=16, L=64, dt=_abi.SS_BF16):
    f = _abi.SS_F32
    return dict(du=FakeT((Bsz, D, L), dt), ddelta=FakeT((Bsz, D, L), dt), dz=FakeT((Bsz, D, L), dt),
                dA=FakeT((D, N), f), dB=FakeT((Bsz, N, L), f), dC=FakeT((Bsz, N, L), f),
                dD=FakeT((D,), f), dbias=FakeT((D,), f))


def test_backward_argument_errors(lib):
    a = _sel_args()  # "y" plays dout
    assert _call_bwd(lib, a, dict(_bwd_grads(), dz=None)) == -1      # z given, dz missing
    assert _call_bwd(lib, a, dict(_bwd_grads(), dD=None)) == -1
    assert _call_bwd(lib, a, dict(_bwd_grads(), dbias=None)) == -1
    assert _call_bwd(lib, a, dict(_bwd_grads(), du=None)) == -1
    assert _call_bwd(lib, a, _bwd_grads(), softplus=3) == -1
    g = _bwd_grads()
    g["du"] = FakeT((2, 8, 63))
    assert _call_bwd(lib, a, g) == -2
    g = _bwd_grads()
    g["ddelta"] = FakeT((2, 8, 64), _abi.SS_F32)
    assert _call_bwd(lib, a, g) == -3
    g = _bwd_grads()
    g["dA"] = FakeT((8, 16), _abi.SS_BF16)
    assert _call_bwd(lib, a, g) == -3
    g = _bwd_grads()
    g["dB"] = FakeT((2, 16, 65), _abi.SS_F32)
    assert _call_bwd(lib, a, g) == -2
    g = _bwd_grads()
    g["dC"] = FakeT((2, 16, 64), _abi.SS_F32, stride=[1024, 1, 16])  # not contiguous
    assert _call_bwd(lib, a, g) == -5
    b = _sel_args(N=32)
    assert _call_bwd(lib, b, _bwd_grads(N=32)) == -5                  # N > 16
    b = _sel_args()
    b["y"] = FakeT((2, 8, 64), _abi.SS_F32)                           # dout dtype
    assert _call_bwd(lib, b, _bwd_grads()) == -3


def test_grouped_bc_argument_errors(lib):
    a = _sel_args(D=12)
    a["B"] = FakeT((2, 5, 16, 64))                         # 12 channels in 5 groups
    a["C"] = FakeT((2, 5, 16, 64))
    assert _call_sel(lib, a) == -2
    a = _sel_args(D=12)
    a["B"] = FakeT((2, 4, 16, 64))
    a["C"] = FakeT((2, 3, 16, 64))                         # B and C disagree
    assert _call_sel(lib, a) == -2
    a = _sel_args(D=12)
    a["B"] = FakeT((2, 4, 16, 64))
    a["C"] = FakeT((2, 4, 16, 64))
    assert _call_bwd(lib, a, _bwd_grads(D=12)) == -5       # backward: shared B, C only


def test_host_buffer_entry_point_rejects_strided_tensors(lib):
    a = _sel_args()
    a["u"] = FakeT((2, 8, 64), stride=[1024, 128, 1])  # rows of 128 with 64 used
    r = {k: v.ref for k, v in a.items()}
    assert lib.ss_selective_scan_fwd_host(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 1, r["y"], r["last"], None) == -5
    b = _sel_args()
    r = {k: v.ref for k, v in b.items()}
    assert lib.ss_selective_scan_fwd_host(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 3, r["y"], r["last"], None) == -1


def _call_fwd_ckpt(lib, a, ck):
    r = {k: (None if v is None else v.ref) for k, v in a.items()}
    return lib.ss_selective_scan_fwd_ckpt(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 1, r["y"], r["last"],
                                          None if ck is None else ck.ref, None)


def _call_bwd_ckpt(lib, a, g, ck):
    r = {k: (None if v is None else v.ref) for k, v in a.items()}
    o = {k: (None if v is None else v.ref) for k, v in g.items()}
    return lib.ss_selective_scan_bwd_ckpt(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"],
                                          r["z"], r["bias"], 1, r["y"],
                                          None if ck is None else ck.ref, o["du"], o["ddelta"],
                                          o["dA"], o["dB"], o["dC"], o["dD"], o["dz"], o["dbias"],
                                          None)


def test_checkpoint_pair_argument_errors(lib):
    f = _abi.SS_F32
    a = _sel_args()  # L = 64: 8 checkpoints per channel
    assert _call_fwd_ckpt(lib, a, None) == -1
    assert _call_fwd_ckpt(lib, a, FakeT((2, 8, 9, 16), f)) == -2          # count of checkpoints
    assert _call_fwd_ckpt(lib, a, FakeT((2, 8, 8, 8), f)) == -2           # 16 states each
    assert _call_fwd_ckpt(lib, a, FakeT((2, 8, 8, 16))) == -3             # fp32 only
    assert _call_fwd_ckpt(lib, a, FakeT((2, 8, 8, 16), f, stride=[2048, 256, 32, 1])) == -5
    assert _call_fwd_ckpt(lib, a, FakeT((2, 8, 8, 16), f, data=0x10004)) == -4  # 16-byte rows
    g = _sel_args()
    g["B"], g["C"] = FakeT((2, 2, 16, 64)), FakeT((2, 2, 16, 64))
    assert _call_fwd_ckpt(lib, g, FakeT((2, 8, 8, 16), f)) == -5          # shared B, C only
    assert _call_bwd_ckpt(lib, a, _bwd_grads(), None) == -1
    assert _call_bwd_ckpt(lib, a, _bwd_grads(), FakeT((2, 8, 7, 16), f)) == -2
    # nothing to scan and no final state asked for: accepted, no device touched
    e = _sel_args(L=0)
    e["last"] = None
    assert _call_fwd_ckpt(lib, e, FakeT((2, 8, 0, 16), f)) == 0
