"""Shape checks of the Python binding (CPU only).

The C calls receive pointers and the sizes read from q and k; the kernels index every
other tensor by those sizes.  So each wrapper refuses a tensor of another shape before
anything reaches the library.  With host tensors a call whose shapes all agree gets
past the shape checks and stops at the first pointer conversion ("must be a CUDA
tensor"), so no call here can launch work on any machine.
"""
import pytest
import torch

from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300.build import build

B, H, NQ, NK, D = 2, 3, 100, 77, 64
F32, U8 = torch.float32, torch.uint8


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()


def z(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def dense_args():
    return dict(q=z(B, H, NQ, D), k=z(B, H, NK, D), v=z(B, H, NK, D), o=z(B, H, NQ, D), lse=z(B, H, NQ, dtype=F32),
                do=z(B, H, NQ, D), dq=z(B, H, NQ, D), dk=z(B, H, NK, D), dv=z(B, H, NK, D))


# one wrong shape per tensor argument
DENSE_BAD = {
    "k": z(B, H, NK, 32), "v": z(B, H, NK + 1, D), "o": z(B, H, NQ - 1, D), "lse": z(B * H, NQ, dtype=F32),
    "do": z(B, H + 1, NQ, D), "dq": z(B, H, NQ, D * 2), "dk": z(B, H, NQ, D), "dv": z(1, H, NK, D),
}

FWD = ("q", "k", "v", "o", "lse")
BWD = ("q", "k", "v", "o", "lse", "do", "dq", "dk", "dv")


def call_dense(name, a):
    if name == "fa_fwd":
        return _lib.fa_fwd(*(a[n] for n in FWD), True)
    if name == "fa_bwd":
        return _lib.fa_bwd(*(a[n] for n in BWD), True)
    if name == "fa_bwd_noalloc":
        return _lib.fa_bwd_noalloc(*(a[n] for n in BWD), True)
    if name == "fa_fwd_window":
        return _lib.fa_fwd_window(*(a[n] for n in FWD), True, 16, -1, 4)
    if name == "fa_bwd_window":
        return _lib.fa_bwd_window(*(a[n] for n in BWD), True, 16, -1, 4, workspace=z(256, dtype=U8))
    if name == "StepGraph":
        return _lib.StepGraph(*(a[n] for n in BWD), True, workspace=z(256, dtype=U8))
    if name == "step_host":
        return _lib.step_host(a["q"], a["k"], a["v"], a["do"], a["o"], a["lse"], a["dq"], a["dk"], a["dv"],
                              z(1024, dtype=U8), True)
    raise AssertionError(name)


DENSE_CALLS = {"fa_fwd": FWD, "fa_fwd_window": FWD, "fa_bwd": BWD, "fa_bwd_noalloc": BWD, "fa_bwd_window": BWD,
               "StepGraph": BWD, "step_host": BWD}


@pytest.mark.parametrize("name", sorted(DENSE_CALLS))
def test_dense_wrappers_pass_matching_shapes(name):
    with pytest.raises(ValueError, match="must be a (CUDA|host) tensor"):
        call_dense(name, dense_args())


@pytest.mark.parametrize("name,arg", [(n, a) for n, args in sorted(DENSE_CALLS.items()) for a in args if a != "q"])
def test_dense_wrappers_refuse_a_mismatched_shape(name, arg):
    a = dense_args()
    a[arg] = DENSE_BAD[arg]
    with pytest.raises(ValueError, match=f"{arg} has shape"):
        call_dense(name, a)


@pytest.mark.parametrize("name", sorted(DENSE_CALLS))
def test_dense_wrappers_refuse_other_ranks(name):
    a = dense_args()
    a["q"] = z(B * H, NQ, D)
    with pytest.raises(ValueError, match=r"must be \[B, H, N, D\]"):
        call_dense(name, a)


def test_forward_fp8_checks_k_and_v_against_q():
    with pytest.raises(ValueError, match="v has shape"):
        _lib.forward_fp8(z(B, H, NQ, D), z(B, H, NK, D), z(B, H, NK + 16, D), True)


def test_quantize_qkv_checks_k_and_v_against_q():
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _lib.quantize_qkv_e4m3(z(B, H, NQ, D), z(B, H, NK, D), z(B, H, NK, D))
    for k, v, msg in ((z(B, H, NK, 128), z(B, H, NK, D), "k has shape"),
                      (z(B, H, NK, D), z(B, H, NK + 16, D), "v has shape"),
                      (z(B, H + 1, NK, D), z(B, H, NK, D), "k has shape"),
                      (z(H, NK, D), z(B, H, NK, D), r"must be \[B, H, N, D\]")):
        with pytest.raises(ValueError, match=msg):
            _lib.quantize_qkv_e4m3(z(B, H, NQ, D), k, v)


def fp8_args():
    ldv = (NK + 15) // 16 * 16
    return dict(q8=z(B, H, NQ, D, dtype=U8), k8=z(B, H, NK, D, dtype=U8), vt8=z(B, H, D, ldv, dtype=U8), ldv=ldv,
                qd=z(1, dtype=F32), kd=z(1, dtype=F32), vd=z(1, dtype=F32), o=z(B, H, NQ, D), lse=z(B, H, NQ, dtype=F32))


def call_fp8(a):
    return _lib.fa_fwd_fp8(a["q8"], a["k8"], a["vt8"], a["ldv"], a["qd"], a["kd"], a["vd"], a["o"], a["lse"], True)


def test_fp8_wrapper_shapes():
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        call_fp8(fp8_args())
    for arg, bad, msg in (("vt8", z(B, H, NK, 80, dtype=U8), "vt8 has shape"),
                          ("k8", z(B, H, NK, 128, dtype=U8), "k has shape"),
                          ("o", z(B, H, NQ, 128), "o has shape"),
                          ("lse", z(B, H, NK, dtype=F32), "lse has shape"),
                          ("vd", z(0, dtype=F32), "v_descale must hold")):
        a = fp8_args()
        a[arg] = bad
        with pytest.raises(ValueError, match=msg):
            call_fp8(a)


TQ, TK, NSEQ = 120, 90, 4


def packed_args():
    cu = torch.tensor([0, 30, 60, 90, 120], dtype=torch.int32)
    cuk = torch.tensor([0, 20, 40, 60, 90], dtype=torch.int32)
    return dict(q=z(TQ, H, D), k=z(TK, H, D), v=z(TK, H, D), o=z(TQ, H, D), lse=z(H, TQ, dtype=F32),
                do=z(TQ, H, D), dq=z(TQ, H, D), dk=z(TK, H, D), dv=z(TK, H, D), cq=cu, ck=cuk)


PACKED_BAD = {
    "k": z(TK, H, 32), "v": z(TK + 1, H, D), "o": z(TQ, H + 1, D), "lse": z(TQ, H, dtype=F32), "do": z(TQ - 1, H, D),
    "dq": z(TQ, H, D * 2), "dk": z(TQ, H, D), "dv": z(TK, 1, D), "ck": torch.zeros(NSEQ, dtype=torch.int32),
}


def call_packed(name, a):
    cu = (a["cq"], a["ck"])
    if name == "fa_fwd_varlen":
        return _lib.fa_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], *cu, 30, 30, True)
    return _lib.fa_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"], a["dv"], *cu,
                              30, 30, True, workspace=z(256, dtype=U8))


PACKED_CALLS = {"fa_fwd_varlen": ("k", "v", "o", "lse", "ck"),
                "fa_bwd_varlen": ("k", "v", "o", "lse", "do", "dq", "dk", "dv", "ck")}


@pytest.mark.parametrize("name", sorted(PACKED_CALLS))
def test_packed_wrappers_pass_matching_shapes(name):
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        call_packed(name, packed_args())


@pytest.mark.parametrize("name,arg", [(n, a) for n, args in sorted(PACKED_CALLS.items()) for a in args])
def test_packed_wrappers_refuse_a_mismatched_shape(name, arg):
    a = packed_args()
    a[arg] = PACKED_BAD[arg]
    want = "cu_seqlens_k has shape" if arg == "ck" else f"{arg} has shape"
    with pytest.raises(ValueError, match=want):
        call_packed(name, a)


def test_packed_wrappers_need_offsets():
    a = packed_args()
    a["cq"] = a["ck"] = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="B \\+ 1 >= 2 offsets"):
        call_packed("fa_fwd_varlen", a)
