"""Helpers for the GPU parity tests: device buffers with canary guard regions."""
import numpy as np
import pytest

GUARD = 64            # floats of canary before and after every device buffer
CANARY = np.float32(-7.7e33)


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


class Guarded:
    """A device float32 (or int32) buffer surrounded by canaries; .t is the payload view."""

    def __init__(self, torch, arr, dtype=np.float32):
        arr = np.ascontiguousarray(arr, dtype=dtype)
        self.shape = arr.shape
        n = arr.size
        tdt = torch.float32 if dtype == np.float32 else torch.int32
        fill = CANARY if dtype == np.float32 else np.int32(-123456789)
        host = np.full(n + 2 * GUARD, fill, dtype=dtype)
        host[GUARD:GUARD + n] = arr.reshape(-1)
        self.full = torch.from_numpy(host).to("cuda")
        self.t = self.full[GUARD:GUARD + n]
        self.fill = fill
        self.n = n

    def numpy(self):
        return self.t.cpu().numpy().reshape(self.shape)

    def guards_intact(self) -> bool:
        h = self.full.cpu().numpy()
        return bool(np.all(h[:GUARD] == self.fill) and np.all(h[GUARD + self.n:] == self.fill))


def empty_guarded(torch, shape, fill=np.nan):
    return Guarded(torch, np.full(shape, fill, dtype=np.float32))


def assert_close(got, want, max_abs, mean_abs=None, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    mx = float(err.max()) if err.size else 0.0
    assert mx <= max_abs, f"{what}: max abs err {mx:.3e} > {max_abs:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    if mean_abs is not None and err.size:
        assert float(err.mean()) <= mean_abs, f"{what}: mean abs err {err.mean():.3e} > {mean_abs:.1e}"
    return mx
