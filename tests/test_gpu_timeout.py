"""The failure path of the d = 64 tensor-core forward (GPU only).

Every wait of that kernel on another warp's progress is bounded.  The testing hook
zeros_debug_walk shortens the bound to about half a millisecond and makes one warp of every CTA
withhold its arrival on the barrier that releases the first S V product, so that the wait for it
runs out.  The call must then report ZEROS_ERR_TIMEOUT through the status word (no fault, no
hang: the other warps leave their loops, in-flight copies and tensor-core work are waited for
and tensor memory is freed), and the next normal call on the same context must be correct.
"""
import numpy as np
import pytest
import torch

import oracle
import zeros_inputs as zi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zs():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import zero_sum_prefix_gb300 as m
    m.load()
    return m


NAMES = ("q", "k", "v", "u", "g1", "gh", "mu", "tau")


def test_walk_wait_timeout_is_reported_and_the_context_recovers(zs):
    w = zi.Workload("timeout", 2, 2, 300, 64, rope=True, seed=4321)
    inp = zi.make(w, "cuda")
    args = [inp[n] for n in NAMES]
    zs.get_status()  # start from a clear status word
    zs.debug_walk(1 << 20, True)
    try:
        zs.fwd(*args, causal=True, rope=True, rope_base=w.rope_base, path="chunk")
        rc = zs.get_status()
    finally:
        zs.debug_walk(0, False)
    assert rc == zs.ZEROS_ERR_TIMEOUT, rc
    o = zs.fwd(*args, causal=True, rope=True, rope_base=w.rope_base, path="chunk")
    assert zs.get_status() == 0
    ref = oracle.forward(*(inp[n].cpu() for n in NAMES), causal=True, rope=True,
                         rope_base=w.rope_base)
    got = o.float().cpu().numpy()
    err = np.abs(got - ref).max() / np.abs(ref).max()
    print(f"error after the timed-out call {err:.3e}")
    assert err <= 1e-2


def test_debug_walk_rejects_negative_limit(zs):
    with pytest.raises(zs.ZerosError):
        zs.debug_walk(-1, False)
