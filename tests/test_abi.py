"""The C-ABI library builds, loads, and exports every function include/ig.h declares.

No GPU is needed: these tests only load the library and exercise argument validation and
host-side fault injection, which return before any CUDA call.
"""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ig():
    from speculative_kv_cache_gb300 import build

    build.build()
    from speculative_kv_cache_gb300 import ig as mod

    return mod


def test_every_declared_function_is_exported(ig):
    names = ig.header_functions()
    assert len(names) >= 20
    for required in ["ig_skew_weights", "ig_speculate", "ig_select", "ig_gather_kv",
                     "ig_sparse_attend", "ig_pool_evict", "ig_pool_create", "ig_pool_destroy",
                     "ig_check"]:
        assert required in names
    lib = ctypes.CDLL(ig.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert hasattr(ig, n), f"binding lacks {n}"


def test_version_and_error_string(ig):
    assert ig.ig_version() == 100
    assert isinstance(ig.ig_last_error(), str)


def test_invalid_arguments_are_rejected_before_any_device_work(ig):
    with pytest.raises(ig.IGError) as e:
        ig.ig_select(0, 1, 1, 8, 16, 32, 0.0, ig.IG_SEL_THRESHOLD, 1.0, 48, 64, None)
    assert e.value.status == ig.IG_ERR_INVALID and "alpha" in str(e.value)
    with pytest.raises(ig.IGError) as e:
        ig.ig_speculate(0, 1, 64, 1, 8, 12, 16, 16, 16, 16, 1.0, 16, None, 256, 1 << 20)
    assert e.value.status == ig.IG_ERR_INVALID and "multiple of 8" in str(e.value)
    with pytest.raises(ig.IGError) as e:
        ig.ig_sparse_attend(0, 1, 1, 96, 8, 1.0, 16, 16, 16, 16, None, None, 16, None, 0)
    assert e.value.status == ig.IG_ERR_INVALID
    with pytest.raises(ig.IGError) as e:
        ig.ig_gather_attend(0, None, 0, 1, 1, 64, 8, 1.0, 16, 16, 16, None, None, 16, None, 0)
    assert e.value.status == ig.IG_ERR_INVALID and "pool" in str(e.value)


def test_decoder_fused_fetch_needs_no_staging_buffers_and_a_fetch_workspace(ig):
    base = dict(layers=2, B=2, H=4, d=64, D=256, k=16, Lcap=64, policy=0, alpha=4.0, cap_frac=1.0,
                score_scale=0.125, rope_theta=0.0, gather_ctas=0, stage_timing=0, fused_select=1)
    staged = ig.ig_decoder_workspace_bytes(ig.DecoderConfig(**base, fused_fetch=0))
    fused = ig.ig_decoder_workspace_bytes(ig.DecoderConfig(**base, fused_fetch=1))
    # the fetch stream's partial attention gets two regions of its own (by layer parity: the
    # compute stream combines layer l's partials while the fetch stream writes layer l+1's)
    assert fused - staged == 2 * ig.ig_gather_attend_workspace_bytes(2, 4, 64, 64)
    # per-head partials of every lane group: (B*H + 256 CTAs) x 32 groups x (d + 2) floats
    assert ig.ig_gather_attend_workspace_bytes(2, 4, 64, 64) >= (8 + 256) * 32 * 66 * 4
    assert ig.ig_gather_attend_workspace_bytes(2, 4, 96, 64) == 0


def test_workspace_sizes(ig):
    assert ig.ig_speculate_workspace_bytes(16, 7168, 56, 38) == 28 * 16 * 56 * 38 * 4
    assert ig.ig_speculate_workspace_bytes(1, 256, 4, 16) == 256
    assert ig.ig_select_workspace_bytes(16, 56) % 256 == 0
    assert ig.ig_attend_workspace_bytes(1, 4, 64, 256) >= 4 * 4 * 66 * 4


def test_injected_pinned_allocation_failure():
    code = ("import os; os.environ['IG_FAULT']='pool_alloc';"
            "from speculative_kv_cache_gb300 import ig;"
            "import sys\n"
            "try:\n ig.ig_pool_create(1, 1, 1, 8, 4)\n"
            "except ig.IGError as e:\n sys.exit(0 if e.status == ig.IG_ERR_OOM else 3)\n"
            "sys.exit(4)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_build_reuses_the_library_only_for_identical_inputs(tmp_path, monkeypatch):
    """The up-to-date check is a hash of the inputs' bytes, flags and tools, not of mtimes."""
    from speculative_kv_cache_gb300 import build

    extra = tmp_path / "extra.cuh"
    extra.write_text("// a header\n")
    real_inputs = build._inputs
    monkeypatch.setattr(build, "_inputs", lambda: real_inputs() + [str(extra)])
    h0 = build.build_hash()
    assert build.build_hash() == h0
    extra.write_text("// a header, edited\n")
    h1 = build.build_hash()
    assert h1 != h0
    os.utime(extra, (0, 0))  # an old mtime does not hide the edit
    assert build.build_hash() == h1
    monkeypatch.setattr(build, "NVCC_FLAGS", build.NVCC_FLAGS + ["-DIG_SOMETHING"])
    assert build.build_hash() != h1
    # a stamp from other inputs never counts as up to date
    monkeypatch.setattr(build, "STAMP", str(tmp_path / "libig.so.sha256"))
    (tmp_path / "libig.so.sha256").write_text(h0 + "\n")
    assert not build.up_to_date(h1)
    assert build.up_to_date(h0) == os.path.exists(build.LIB)


def test_injected_svd_non_convergence():
    """IG_FAULT=svd_noconverge leaves the Jacobi iteration no sweeps: ig_skew_weights (a host
    call) must report IG_ERR_NUMERIC, and the same call without the fault must succeed."""
    code = ("import os, sys\n"
            "import numpy as np\n"
            "from speculative_kv_cache_gb300 import ig\n"
            "D, H, d, Ns = 32, 2, 8, 16\n"
            "g = np.random.default_rng(0)\n"
            "X = g.standard_normal((Ns, D)).astype(np.float16)\n"
            "W = (0.1 * g.standard_normal((D, H * d))).astype(np.float16)\n"
            "A = np.zeros((H, d, d), np.float32); cols = np.zeros((H, 4), np.int32)\n"
            "args = (D, H, d, 0.5, 0.0, X, Ns, W, W, None, 0, A, None, None, None, cols)\n"
            "if os.environ.get('IG_FAULT'):\n"
            "    try:\n"
            "        ig.ig_skew_weights(*args)\n"
            "    except ig.IGError as e:\n"
            "        sys.exit(0 if e.status == ig.IG_ERR_NUMERIC and 'converge' in str(e) else 3)\n"
            "    sys.exit(4)\n"
            "sys.exit(0 if ig.ig_skew_weights(*args) == 4 else 5)\n")
    for fault in ("svd_noconverge", ""):
        env = dict(os.environ, IG_FAULT=fault)
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, env=env)
        assert r.returncode == 0, (fault, r.returncode, r.stderr)
