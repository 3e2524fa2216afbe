"""Shared helpers of the GPU parity tests (comparison rules and oracle runs)."""
import numpy as np
import torch

# fp32 state tolerance: relative 1e-6 with an absolute floor far below any
# value the workloads produce (v ~ 1e-11 at sigma = 1e-4 is still normal).
STATE_RTOL = 1e-6
STATE_ATOL = 1e-30


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16/f16 tensor (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def host(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy: fp32 as float32, bf16/f16 as raw uint16 bits."""
    if t.dtype == torch.float32:
        return t.detach().cpu().numpy().copy()
    return bits16(t)


def ordered16(bits: np.ndarray) -> np.ndarray:
    """16-bit float patterns -> integers in numeric order (one step = one ulp)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b)


def assert_state_close(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    assert got.shape == want.shape, what
    ok = np.abs(got.astype(np.float64) - want) <= STATE_RTOL * np.abs(want.astype(np.float64)) + STATE_ATOL
    ok |= (got == want) | (np.isnan(got) & np.isnan(want))
    if not ok.all():
        i = np.flatnonzero(~ok)[:5]
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} elements beyond 1e-6 rel, e.g. idx {i} "
                             f"got {got[i]} want {want[i]}")


def assert_out_close(got: np.ndarray, want: np.ndarray, fmt: str, what: str = "") -> None:
    """Compute-dtype outputs: within 1 ulp (16-bit formats) / the state rule (fp32)."""
    if fmt == "f32":
        assert_state_close(got, want, what)
        return
    d = np.abs(ordered16(got) - ordered16(want))
    if d.max(initial=0) > 1:
        i = np.flatnonzero(d > 1)[:5]
        raise AssertionError(f"{what}: {np.count_nonzero(d > 1)} outputs beyond 1 ulp, e.g. idx {i}")


def np_grad(t: torch.Tensor) -> np.ndarray:
    """Gradient tensor -> oracle storage (fp32 floats or 16-bit patterns)."""
    return host(t)
