"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks return their status codes without launching anything."""
import ctypes
import os
import re

import pytest

import mixture_experts_layer_topk_gb300 as M

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = M.load()
    names = declared_symbols()
    assert "moe_router_topk" in names and "moe_permute_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    for n in M.EXPORTED:
        assert n in names


def test_library_is_built_for_sm103a():
    stamp = os.path.join(ROOT, "mixture_experts_layer_topk_gb300", "_build", "stamp")
    M.load()
    assert os.path.exists(stamp)
    from mixture_experts_layer_topk_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH


def cfg(**kw):
    base = dict(T=256, H=128, E=8, k=2, F=256, F_shared=0, score_fn=0, renorm=1, gate_scale=1.0, n_group=1,
                topk_group=1, group_score=0, align=128, reserved=0)
    base.update(kw)
    return M.MoeConfig(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(), 0),
    (dict(k=9), 1), (dict(k=0), 1), (dict(T=-1), 1), (dict(score_fn=2), 1), (dict(align=0), 1),
    (dict(E=8, n_group=3), 1), (dict(E=16, k=8, n_group=4, topk_group=1), 1), (dict(n_group=2, topk_group=3), 1),
    (dict(H=192), 2), (dict(F=200), 2), (dict(F_shared=64), 2), (dict(E=512, k=2), 2), (dict(k=33, E=64), 2),
])
def test_config_checks(kw, status):
    lib = M.load()
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg(**kw)), ctypes.byref(n)) == status
    if status == 0:
        assert n.value > 0
        R = ctypes.c_int64()
        assert lib.moe_max_rows(ctypes.byref(cfg(**kw)), ctypes.byref(R)) == 0
        assert R.value == 256 * 2 + 8 * 127


def test_null_and_misaligned_pointers_rejected_before_launch():
    lib = M.load()
    c = cfg()
    nul = [None] * 10
    assert lib.moe_router_topk(ctypes.byref(c), *nul, None) == 1
    assert lib.moe_permute(ctypes.byref(c), *([None] * 9), None) == 1
    fake = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1002)
    # misaligned bf16 buffer
    assert lib.moe_unpermute_combine(ctypes.byref(c), odd, fake, fake, None, fake, None) == 1
    # align != 128 is not supported by the grouped GEMM
    c1 = cfg(align=1)
    args = [fake] * 8 + [None] * 6 + [fake]
    assert lib.moe_grouped_swiglu_mlp(ctypes.byref(c1), *args, None) == 2
    # missing workspace
    assert lib.moe_permute(ctypes.byref(c), *([fake] * 8), None, None) == 3


def test_status_strings():
    lib = M.load()
    for s in range(7):
        assert lib.moe_status_string(s)
