"""The C ABI library loads and exports what include/moe.h declares; host-side
validation works without a GPU (no call here reaches a kernel)."""
import ctypes
import math
import os
import re

import pytest

import routing_permute_grouped_router_gb300 as pkg
from oracle import moe_oracle as O
from routing_permute_grouped_router_gb300 import build as B
from routing_permute_grouped_router_gb300 import workload as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pkg.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(pkg._SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for i, s in enumerate(pkg.STATUS):
        assert lib.moe_status_string(i).decode() == s


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_capacity_matches_oracle(lib, name):
    s = W.WORKLOADS[name]
    C = pkg.moe_capacity(pkg.config_of(s))
    ref = O.capacity(s.T, s.k, s.E, s.capacity_factor)
    assert C == (-1 if ref is None else ref)


def test_capacity_override_and_factor_rounding(lib):
    assert pkg.moe_capacity(pkg.config(100, 256, 256, 8, 2, 1.25, capacity=0)) == 0
    assert pkg.moe_capacity(pkg.config(100, 256, 256, 8, 2, 1.25, capacity=7)) == 7
    for cf in (0.3, 1.1, 1.7, 2.0, 0.01):
        for T in (1, 7, 333, 4096):
            got = pkg.moe_capacity(pkg.config(T, 256, 256, 6, 2, cf))
            assert got == O.capacity(T, 2, 6, cf)


def test_max_rows_bounds_every_layout(lib):
    for (T, E, k, cap) in [(300, 4, 2, -1), (300, 4, 2, 0), (300, 4, 2, 5), (4096, 8, 2, 1280), (1, 128, 8, -1)]:
        cfg = pkg.config(T, 256, 256, E, k, 0.0, capacity=cap)
        R = pkg.moe_max_rows(cfg)
        assert R % 128 == 0
        C = None if cap < 0 else cap
        worst = 0
        # worst case: counts as uneven as the capacity allows
        per = [0] * E
        left = T * k
        for e in range(E):
            take = min(left, C if C is not None else left, T)
            per[e] = take
            left -= take
        worst = sum(128 * math.ceil(c / 128) for c in per)
        assert R >= worst
        assert R >= (min(T * k, E * (C if C is not None else T * k)))


def test_workspace_sizes_positive(lib):
    for s in W.WORKLOADS.values():
        cfg = pkg.config_of(s)
        assert pkg.moe_workspace_size(cfg, 0) > 0
        assert pkg.moe_workspace_size(cfg, 1) > 0


@pytest.mark.parametrize("kw,err", [
    (dict(T=-1), "MOE_ERR_SHAPE"), (dict(E=0), "MOE_ERR_SHAPE"), (dict(k=0), "MOE_ERR_SHAPE"),
    (dict(k=9, E=16), "MOE_ERR_SHAPE"), (dict(k=5, E=4), "MOE_ERR_SHAPE"), (dict(E=129), "MOE_ERR_SHAPE"),
    (dict(d_model=100), "MOE_ERR_SHAPE"), (dict(d_ff=320), "MOE_ERR_SHAPE"), (dict(dtype=7), "MOE_ERR_DTYPE"),
    (dict(aux_loss_coeff=-0.01), "MOE_ERR_INVALID_ARG"), (dict(aux_loss_coeff=float("nan")), "MOE_ERR_INVALID_ARG"),
])
def test_invalid_configs_rejected_on_host(lib, kw, err):
    base = dict(T=64, d_model=256, d_ff=256, E=4, k=2, capacity_factor=1.0, capacity=-1, dtype=pkg.MOE_BF16,
                aux_loss_coeff=0.0)
    base.update(kw)
    cfg = pkg.MoeConfig(*[base[n] for n, _ in pkg.MoeConfig._fields_])
    with pytest.raises(pkg.MoeError) as ei:
        pkg.moe_max_rows(cfg)
    assert err in str(ei.value)


def test_null_and_misaligned_pointers_rejected_before_any_launch(lib):
    cfg = pkg.config(64, 256, 256, 4, 2, 1.0)
    n0 = lib.moe_launch_count()
    rc = lib.moe_permute(ctypes.byref(cfg), None, None, None, None, None, None)
    assert pkg.STATUS[rc] == "MOE_ERR_INVALID_ARG"
    rc = lib.moe_permute(ctypes.byref(cfg), 0x1001, 0x1000, 0x1000, 0x1000, 0x2000, None)
    assert pkg.STATUS[rc] == "MOE_ERR_ALIGNMENT"
    rc = lib.moe_router_topk(ctypes.byref(cfg), *([0x1000] * 11), 0x1000, 16, None)
    assert pkg.STATUS[rc] == "MOE_ERR_WORKSPACE"
    rc = lib.moe_layer_fwd(None, None, None, None, None, None, 0, None)
    assert pkg.STATUS[rc] == "MOE_ERR_INVALID_ARG"
    assert lib.moe_launch_count() == n0


def test_kernel_names(lib):
    n = lib.moe_kernel_kinds()
    names = [lib.moe_kernel_name(i).decode() for i in range(n)]
    assert "gemm_up_swiglu" in names and "permute" in names and len(set(names)) == n
    assert lib.moe_kernel_name(n) is None


def test_recompute_workspace_is_larger_and_training_flag_checked(lib):
    cfg = pkg.config(1000, 256, 512, 8, 2, 1.25)
    w1, w2 = pkg.moe_workspace_size(cfg, 1), pkg.moe_workspace_size(cfg, 2)
    R = pkg.moe_max_rows(cfg)
    assert w2 - w1 >= 3 * R * 512 * 2  # a, b, h of the recompute
    with pytest.raises(pkg.MoeError):
        pkg.moe_workspace_size(cfg, 3)


def test_nvtx_switch_is_host_only(lib):
    # toggling the NVTX ranges touches no device: it works without a GPU
    n0 = lib.moe_launch_count()
    assert lib.moe_nvtx_enable(1) == 0
    assert lib.moe_nvtx_enable(0) == 0
    assert lib.moe_launch_count() == n0
