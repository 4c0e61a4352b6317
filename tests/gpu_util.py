"""Helpers for the GPU parity tests: device buffers from NumPy and back (no method arithmetic)."""
import numpy as np
import torch

DEV = "cuda:0"


def dev(a: np.ndarray) -> torch.Tensor:
    """Device copy of a NumPy array (fp16 stays fp16, int32 stays int32)."""
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def empty(shape, dtype) -> torch.Tensor:
    return torch.empty(shape, dtype=dtype, device=DEV)


def workspace(nbytes: int) -> torch.Tensor:
    # torch's caching allocator returns 256-byte (or better) aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=DEV)


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def score_ok(s_gpu, s_ora, L):
    """Scores within 1e-3 of the per-head largest |s| (the stated relative tolerance)."""
    B, H, _ = s_ora.shape
    worst = 0.0
    for b in range(B):
        l = int(L[b])
        if l == 0:
            continue
        ref = s_ora[b, :, :l]
        scale = np.maximum(np.abs(ref).max(axis=1), 1e-30)
        err = (np.abs(s_gpu[b, :, :l].astype(np.float64) - ref).max(axis=1)) / scale
        worst = max(worst, float(err.max()))
        assert np.all(np.isneginf(s_gpu[b, :, l:])), "slots past L_valid must score -inf"
    return worst


def index_sets_ok(idx_gpu, cnt_gpu, s_ora, L, alpha, band=1e-3):
    """GPU sets equal the oracle's threshold sets except tokens within `band` of the threshold.

    Returns the number of exempt disagreements.
    """
    B, H, _ = s_ora.shape
    exempt = 0
    for b in range(B):
        l = int(L[b])
        for h in range(H):
            got = set(idx_gpu[b, h, :cnt_gpu[b, h]].tolist())
            assert list(idx_gpu[b, h, :cnt_gpu[b, h]]) == sorted(got), "indices must ascend"
            s = s_ora[b, h, :l]
            if l == 0:
                assert not got
                continue
            thr = s.max() - alpha
            want = set(np.nonzero(s > thr)[0].tolist()) if np.isfinite(alpha) else set(range(l))
            for t in got ^ want:
                assert 0 <= t < l
                assert abs(s[t] - thr) <= band, f"token {t} of ({b},{h}) differs, gap {s[t] - thr}"
                exempt += 1
    return exempt
