"""ig_speculate_static: speculation for callers that cannot allocate device memory.

Some programs that embed this library reserve all device memory for their own allocator
up front, or must not pay the synchronisation a cudaMalloc can bring, so they cannot hand
ig_speculate a workspace.  ig_speculate_static keeps its scratch in a fixed 4 MiB array
inside the library instead.  These tests call it through the C ABI and check that its output
equals ig_speculate's (with a caller workspace) bit for bit on two calls in a row (both run
the same kernels with the same grids), that a call after the first one on a device leaves the
device's free memory unchanged, and that a request too large for the fixed array is refused
with a clear error.  The file is named so that pytest collects it last.
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


def _case(w, Lcap, layer):
    K, _ = synth.pool_layer(w, layer, cap=Lcap)
    cols = synth.skewed_columns(w, layer)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")  # noqa: E731
    L = np.array([min(w.prompt, Lcap) - (3 * b) % 17 for b in range(w.batch)], dtype=np.int32)
    return dict(x=dev(synth.layer_inputs(w, layers=layer)[layer - 1]), W=dev(synth.skewed_partial_weight(w, layer).T),
                Kpart=dev(ora.partial_key_cache(K, cols)), L=dev(L), Lh=L)


def _both(ig, w, Lcap, c):
    B, D, H, k = w.batch, w.hidden, w.heads, w.k
    scale = 1.0 / math.sqrt(w.head_dim)
    s_ref = torch.empty((B, H, Lcap), dtype=torch.float32, device="cuda:0")
    q_ref = torch.empty((B, H, k), dtype=torch.float32, device="cuda:0")
    ws = torch.empty(ig.ig_speculate_workspace_bytes(B, D, H, k), dtype=torch.uint8, device="cuda:0")
    ig.ig_speculate(None, B, D, H, k, Lcap, c["x"], c["W"], c["Kpart"], c["L"], scale, s_ref, q_ref, ws,
                    ws.numel())
    s_st = torch.full((B, H, Lcap), float("nan"), dtype=torch.float32, device="cuda:0")
    q_st = torch.full((B, H, k), float("nan"), dtype=torch.float32, device="cuda:0")
    ig.ig_speculate_static(None, B, D, H, k, Lcap, c["x"], c["W"], c["Kpart"], c["L"], scale, s_st, q_st)
    ig.ig_check()
    return s_ref.cpu().numpy(), q_ref.cpu().numpy(), s_st.cpu().numpy(), q_st.cpu().numpy()


def _same(ref, got, L):
    assert np.array_equal(got, ref)
    for b, l in enumerate(L):
        assert np.all(np.isneginf(got[b, :, l:]))


def test_static_scratch_matches_workspace_version_on_two_calls(ig):
    # two calls in a row with different shapes: the second reuses (and overwrites) the scratch
    # the first one left behind
    shapes = [(synth.WORKLOADS["opt-30b"], 2048, 1),
              (synth.scaled(synth.WORKLOADS["opt-6.7b"], name="na", batch=3, heads=7, hidden=1024,
                            prompt=500, gen=0), 504, 2)]
    for w, Lcap, layer in shapes:
        c = _case(w, Lcap, layer)
        s_ref, q_ref, s_st, q_st = _both(ig, w, Lcap, c)
        _same(s_ref, s_st, c["Lh"])
        assert np.array_equal(q_st, q_ref)


def test_static_scratch_call_allocates_no_device_memory(ig):
    w = synth.scaled(synth.WORKLOADS["opt-6.7b"], name="na2", batch=2, heads=5, hidden=640,
                     prompt=300, gen=0)
    Lcap = 320
    c = _case(w, Lcap, 1)
    B, D, H, k = w.batch, w.hidden, w.heads, w.k
    scores = torch.empty((B, H, Lcap), dtype=torch.float32, device="cuda:0")
    q = torch.empty((B, H, k), dtype=torch.float32, device="cuda:0")
    args = (None, B, D, H, k, Lcap, c["x"], c["W"], c["Kpart"], c["L"], 0.125, scores, q)
    # the first call on the device looks up the scratch address and loads the kernels
    ig.ig_speculate_static(*args)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    ig.ig_speculate_static(*args)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    ig.ig_check()
    assert free_after == free_before


def test_static_scratch_refuses_requests_beyond_its_size(ig):
    # 28 splits x B x H*k floats beyond 4 MiB: 28 * 64 * 56 * 38 * 4 = 15 MB
    B, D, H, k, Lcap = 64, 7168, 56, 38, 8
    assert ig.ig_speculate_workspace_bytes(B, D, H, k) > 4 << 20
    t = torch.zeros(16, dtype=torch.float32, device="cuda:0")
    with pytest.raises(ig.IGError) as e:
        ig.ig_speculate_static(None, B, D, H, k, Lcap, t, t, t, t, 1.0, t, None)
    assert e.value.status == ig.IG_ERR_CAPACITY and "static" in str(e.value)
