"""The allocation-free router entry point, moe_router_topk_noalloc.

Some callers cannot allocate device memory: a plugin whose host program owns
every allocation, a service whose memory budget is fixed at start-up, or a
latency-critical loop that cannot pay for the implicit device synchronisation
of cudaMalloc/cudaFree.  moe_router_topk_noalloc serves them from a static
device array that the library holds for the life of the process.  It runs
the same router kernels as moe_router_topk, which takes a workspace from the
caller, so these tests call it twice in a row through the C ABI and require
each result to equal moe_router_topk's bit for bit: the integer routing state,
the gates and the probabilities (the tolerance the other tests allow gates and
probabilities, 1e-5, is not needed here).
"""
import ctypes

import pytest
import torch

import routing_permute_grouped_router_gb300 as pkg
from routing_permute_grouped_router_gb300 import workload as W

pytestmark = pytest.mark.gpu

LS = W.LayerShape
SHAPES = [
    LS("top2_e8", 1000, 256, 512, 8, 2, 1.25, W.BF16),
    LS("zipf_e64", 2000, 256, 256, 64, 2, 1.0, W.BF16, zipf_s=1.1),
    LS("dropless_e32_k4", 1500, 512, 256, 32, 4, 0.0, W.BF16, zipf_s=1.3),
    W.WORKLOADS["switch_tiny_f32"],
    # the largest layer at full size: tensor-core router with its W_r parts in the static array
    W.WORKLOADS["dropless_e32_bf16"],
]


@pytest.fixture(scope="module", autouse=True)
def built():
    from routing_permute_grouped_router_gb300 import build

    build.build()
    pkg.lib()
    torch.cuda.set_device(0)
    pkg.moe_get_device_error(clear=True)


def _outputs(cfg, device="cuda"):
    R = pkg.moe_max_rows(cfg)
    i32, f32 = dict(dtype=torch.int32, device=device), dict(dtype=torch.float32, device=device)
    # fill with junk so that anything left unwritten shows up as a difference
    return dict(ids=torch.full((cfg.T, cfg.k), -7, **i32), gates=torch.full((cfg.T, cfg.k), -7.0, **f32),
                probs=torch.full((cfg.T, cfg.E), -7.0, **f32), slot=torch.full((cfg.T, cfg.k), -7, **i32),
                row_of=torch.full((cfg.T, cfg.k), -7, **i32), src_token=torch.full((R,), -7, **i32),
                counts=torch.full((cfg.E,), -7, **i32), offsets=torch.full((cfg.E + 1,), -7, **i32))


def _args(o):
    return (o["ids"], o["gates"], o["probs"], o["slot"], o["row_of"], o["src_token"], o["counts"], o["offsets"])


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_noalloc_router_matches_workspace_router_on_two_calls_in_a_row(shape):
    wl = W.make(shape, micro_batches=1, with_dy=False)
    cfg = pkg.config_of(shape)
    x = wl.x[0].torch("cuda")
    W_r = torch.from_numpy(wl.W_r).cuda()
    bias = None if wl.bias is None else torch.from_numpy(wl.bias).cuda()

    ref = _outputs(cfg)
    ws = pkg.workspace(cfg, 0)
    pkg.moe_router_topk(cfg, x, W_r, bias, *_args(ref), ws)
    torch.cuda.synchronize()
    rows = int(ref["offsets"][-1].item())

    for call in range(2):
        got = _outputs(cfg)
        pkg.moe_router_topk_noalloc(cfg, x, W_r, bias, *_args(got))
        torch.cuda.synchronize()
        code, detail = pkg.moe_get_device_error(clear=True)
        assert code == 0, (call, code, detail)
        for n in ("ids", "slot", "row_of", "counts", "offsets"):
            assert torch.equal(got[n], ref[n]), (call, n)
        assert torch.equal(got["src_token"][:rows], ref["src_token"][:rows]), call
        assert torch.equal(got["gates"], ref["gates"]), call
        assert torch.equal(got["probs"], ref["probs"]), call


def test_noalloc_router_rejects_layers_beyond_its_scratch():
    # E = 128, k = 8 and 60,000 tokens need 2 * 128 * 8 * 938 * 4 bytes of
    # histograms, more than MOE_NOALLOC_SCRATCH_BYTES (4 MiB): refused on the
    # host, before anything is launched.
    cfg = pkg.config(60000, 256, 256, 128, 8, 1.0)
    lib = pkg.lib()
    n0 = lib.moe_launch_count()
    dummy = torch.empty(64, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    rc = lib.moe_router_topk_noalloc(ctypes.byref(cfg), p, p, None, p, p, None, p, p, p, p, p, None)
    assert pkg.STATUS[rc] == "MOE_ERR_WORKSPACE"
    assert lib.moe_launch_count() == n0
