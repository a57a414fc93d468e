"""Parity of the expert co-selection matrix (moe_coselect) with the oracle: bit-exact
integer counts on the oracle's routing indices, small cases and the 256-expert clustered
workload at full size (the workload built to make co-selection correlated)."""
import numpy as np
import pytest
import torch

import synth
import parity as P

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["small-top2-cap1.0", "small-hybrid-top8", "small-clusters-cap1.0",
                                  "small-max-e256-k8", "top2-e256-clusters-cap1.0",
                                  "hybrid-top8-e128-temp0.2", "small-dense-e8",
                                  "small-dense-e12-cap0.5"])
def test_coselect_matches_oracle(name, moe_lib, cuda_device):
    moe = moe_lib
    cfg = synth.get(name)
    inp = synth.make_inputs(cfg, with_dy=False)
    npin = P.np_inputs(inp)
    idx = P.O.route(npin["x"], npin["Wg"], npin["bg"], cfg.k, cfg.temperature)["idx"]
    c = moe.config_from(cfg)
    H = torch.full((cfg.E, cfg.E), -1, dtype=torch.int32, device="cuda")
    moe.coselect(c, P.dev_i32(idx), H)
    moe.get_error()
    ref = P.O.coselection(idx, cfg.E)
    assert (H.cpu().numpy() == ref).all()
    assert int(H.diagonal().sum()) == cfg.T * cfg.k


def test_coselect_rejects_bad_ids(moe_lib, cuda_device):
    moe = moe_lib
    c = moe.make_config(4, 64, 8, 2, 64)
    idx = torch.tensor([[0, 1], [2, 2], [9, 3], [4, 5]], dtype=torch.int32, device="cuda")
    H = torch.zeros(8, 8, dtype=torch.int32, device="cuda")
    moe.coselect(c, idx, H)
    with pytest.raises(moe.MoeError) as ei:
        moe.get_error()
    assert ei.value.status == moe.MOE_ERR_DEVICE_BOUNDS
    Hc = H.cpu().numpy()
    assert Hc[0, 1] == 1 and Hc[4, 5] == 1 and Hc[2, 2] == 1 and Hc[3, 3] == 1


def test_coselect_dense_rejects_non_identity(moe_lib, cuda_device):
    """k = E > 8: idx must be the identity; a token that breaks it is flagged and not counted."""
    moe = moe_lib
    T, E = 5, 12
    c = moe.make_config(T, 64, E, E, 64)
    idx = torch.arange(E, dtype=torch.int32, device="cuda").repeat(T, 1)
    idx[3, 4] = 5
    H = torch.zeros(E, E, dtype=torch.int32, device="cuda")
    moe.coselect(c, idx, H)
    with pytest.raises(moe.MoeError) as ei:
        moe.get_error()
    assert ei.value.status == moe.MOE_ERR_DEVICE_BOUNDS
    ref = np.triu(np.full((E, E), T - 1, dtype=np.int64))
    assert (H.cpu().numpy() == ref).all()
