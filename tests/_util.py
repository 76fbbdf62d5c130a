"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

TOL = {"bf16": 2e-2, "f32": 1e-4}


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, np.float64)


def assert_close(name, got, exp, tol):
    """max|got - exp| <= tol * max|exp| over the whole tensor."""
    g, e = to64(got), to64(exp)
    assert g.shape == e.shape, f"{name}: shape {g.shape} != {e.shape}"
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    scale = np.abs(e).max() if e.size else 0.0
    err = np.abs(g - e).max() if e.size else 0.0
    assert err <= tol * scale or (scale == 0.0 and err == 0.0), \
        f"{name}: max|gpu-ref| = {err:.4e} > {tol} * max|ref| = {tol * scale:.4e}"


def assert_routing_equal(saved, ref, T):
    """Bit-exact comparison of the integer routing state."""
    for name in ("ids", "slot", "row_of", "counts", "offsets"):
        got = saved[name].cpu().numpy()
        exp = np.asarray(ref[name])
        if name in ("ids", "slot", "row_of"):
            got = got[:T]
        assert got.shape == exp.shape, f"{name}: shape {got.shape} != {exp.shape}"
        if not np.array_equal(got, exp):
            bad = np.argwhere(got != exp)[:5]
            raise AssertionError(f"{name} differs at {bad.tolist()}: gpu {got[tuple(bad.T)]} ref {exp[tuple(bad.T)]}")
    rows = int(ref["offsets"][-1])
    got_src = saved["src_token"].cpu().numpy()[:rows]
    assert np.array_equal(got_src, ref["src_token"]), "src_token differs"


def check_no_device_error():
    import routing_permute_grouped_router_gb300 as pkg

    code, detail = pkg.moe_get_device_error(clear=True)
    assert code == 0, f"device error word: code {code} detail {detail:#x}"
