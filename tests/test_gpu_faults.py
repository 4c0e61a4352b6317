"""Failure detection on the GPU without faulting it.

A bounded in-kernel wait is made to run out by setting its iteration limit to 0
(ig_set_wait_limit): the score kernels' first wait for their staged copies then gives up at
once, the kernel records IG_DEVERR_TIMEOUT, lets its copies in flight land (with the default
limit) and leaves, and ig_check reports IG_ERR_TIMEOUT.  Nothing traps, nothing hangs, and the
context stays usable: with the default limit restored the same call succeeds and gives the
same scores as before.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import infinigen as ora  # noqa: E402
from speculative_kv_cache_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ig():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for the -m gpu tests")
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig as mod

    return mod


def test_bounded_wait_runs_out_reports_timeout_and_leaves_the_context_usable(ig):
    w = synth.scaled(synth.WORKLOADS["opt-30b"], name="faults", batch=2, heads=4, hidden=512, prompt=1000, gen=0)
    B, D, H, d, k, Lcap = w.batch, w.hidden, w.heads, w.head_dim, w.k, 1024
    K, _ = synth.pool_layer(w, 1, cap=Lcap)
    cols = synth.skewed_columns(w, 1)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")  # noqa: E731
    x = dev(synth.layer_inputs(w, layers=1)[0])
    W = dev(synth.skewed_partial_weight(w, 1).T)
    Kpart = dev(ora.partial_key_cache(K, cols))
    L = dev(np.array([1000, 777], dtype=np.int32))
    scale = 1.0 / math.sqrt(d)
    ws = torch.empty(max(ig.ig_speculate_workspace_bytes(B, D, H, k),
                         ig.ig_speculate_select_workspace_bytes(B, D, H, d, k, 0)), dtype=torch.uint8,
                     device="cuda:0")
    scores = torch.empty((B, H, Lcap), dtype=torch.float32, device="cuda:0")
    idx = torch.empty((B, H, Lcap), dtype=torch.int32, device="cuda:0")
    cnt = torch.empty((B, H), dtype=torch.int32, device="cuda:0")

    def speculate():
        ig.ig_speculate(None, B, D, H, k, Lcap, x, W, Kpart, L, scale, scores, None, ws, ws.numel())

    def speculate_select():
        ig.ig_speculate_select(None, B, D, H, d, k, Lcap, x, W, None, None, 0.0, Kpart, L, scale, 4.0, idx, cnt,
                               None, None, None, ws, ws.numel())

    ig.ig_check()  # a clean error word to start from
    speculate()
    ig.ig_check()
    before = scores.cpu().numpy().copy()
    try:
        ig.ig_set_wait_limit(0)
        for call in (speculate, speculate_select):
            call()
            with pytest.raises(ig.IGError) as e:
                ig.ig_check()
            assert e.value.status == ig.IG_ERR_TIMEOUT, str(e.value)
            ig.ig_check()  # ig_check cleared the word: nothing left to report
    finally:
        ig.ig_set_wait_limit(-1)
    scores.fill_(float("nan"))
    speculate()
    ig.ig_check()
    assert np.array_equal(scores.cpu().numpy(), before)
    speculate_select()
    ig.ig_check()
