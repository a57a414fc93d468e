"""Routing with exactly tied logits. Small-integer x and Wg (exact in bf16) make every logit an
integer that the fp32 accumulation holds exactly, so logits tie exactly on the GPU and in the
fp64 oracle alike. The selection (ties to the lower expert id, slots in order of logit) is
then compared bit-exact on every token, with no near-tie exclusion. The narrow cases put more
than 16 experts at the 8th logit of many tokens, the wide ones spread the logits so that ties
fall inside and at the edge of the top k. Both routers are covered: the tensor-core one (bf16,
d % 64 = 0) and the CUDA-core one (fp32, or d % 64 != 0)."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu

# name: (T, d, E, k, temperature, x values, Wg values, Wg density, dtype). The tensor-core
# router takes bf16 with d % 64 = 0; fp32, or d % 64 != 0, goes to the CUDA-core router.
CASES = {
    "ties-e64-k8-wide": (2048, 128, 64, 8, 0.2, (-2, -1, 0, 1, 2), (-1, 0, 1), 1.0, "bf16"),
    "ties-e256-k8-narrow": (1024, 64, 256, 8, 0.5, (0, 1), (0, 1), 0.05, "bf16"),
    "ties-e16-k8-narrow": (1500, 64, 16, 8, 1.0, (-1, 0, 1), (0, 1), 0.1, "bf16"),
    "ties-e128-k2-wide": (2048, 128, 128, 2, 1.0, (-2, -1, 0, 1, 2), (-1, 0, 1), 1.0, "bf16"),
    "ties-e200-k4-narrow": (1024, 64, 200, 4, 1.0, (0, 1), (0, 1), 0.05, "bf16"),
    "ties-f32-e64-k8-narrow": (1024, 64, 64, 8, 0.5, (0, 1), (0, 1), 0.1, "f32"),
    "ties-bf16-d40-e32-k3": (1024, 40, 32, 3, 1.0, (-1, 0, 1), (0, 1), 0.2, "bf16"),
}


def _inputs(T, d, E, xv, wv, density, seed):
    rng = np.random.default_rng(seed)
    x = rng.choice(np.array(xv, dtype=np.float32), size=(T, d))
    Wg = rng.choice(np.array(wv, dtype=np.float32), size=(E, d)) * (rng.random((E, d)) < density)
    return x, Wg.astype(np.float32)


@pytest.mark.parametrize("name", list(CASES))
def test_route_exact_ties(name, moe_lib, cuda_device):
    moe = moe_lib
    T, d, E, k, temp, xv, wv, density, dtype = CASES[name]
    x, Wg = _inputs(T, d, E, xv, wv, density, seed=11)
    fwd = P.O.route(x.astype(np.float64), Wg.astype(np.float64), None, k, temp)
    z = fwd["z"]
    assert (z == np.round(z)).all() and np.abs(z).max() < 2 ** 20      # integer logits, exact in fp32
    # the cases exercise ties: some token's k-th and (k+1)-th logits are equal
    kth = -np.sort(-z, axis=1)
    assert (kth[:, k - 1] == kth[:, k]).any()
    cfg = synth.LayerConfig(name=name, T=T, d=d, E=E, k=k, d_ff=64, capacity_factor=None, temperature=temp,
                            dtype=dtype)
    c = moe.config_from(cfg)
    b = moe.alloc_buffers(c, backward=False)
    act = torch.bfloat16 if dtype == "bf16" else torch.float32
    xd = torch.as_tensor(x).to(act).cuda()
    Wd = torch.as_tensor(Wg).to(act).cuda()
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    moe.route(c, xd, Wd, None, b, logits=logits)
    moe.get_error()
    assert np.array_equal(logits.cpu().double().numpy(), z)
    idx = b["idx"].cpu().numpy()
    bad = (idx != fwd["idx"]).any(axis=1)
    assert not bad.any(), f"{bad.sum()} tokens differ, first {np.flatnonzero(bad)[:5]}"
    w = b["w"].cpu().double().numpy()
    P.assert_close("w", w, fwd["w"], 1e-5)
    assert (b["counts"].cpu().numpy() == fwd["counts"]).all()
