"""The oracle's bf16 and fp16 casts on every one of the 2^32 fp32 bit
patterns, against torch's own round-to-nearest-even conversions (a library
routine, not the oracle). NaN in must give NaN out; payloads may differ."""
import numpy as np
import pytest
import torch

NAN_CHUNKS = {31, 63}  # chunks of 2^26 patterns holding exponent-all-ones inputs


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_cast_exhaustive_vs_torch(orc, fmt):
    tdt = torch.bfloat16 if fmt == "bf16" else torch.float16
    exp_mask, man_mask = (0x7f80, 0x007f) if fmt == "bf16" else (0x7c00, 0x03ff)
    n = 1 << 26
    ramp = np.arange(n, dtype=np.uint32)
    for chunk in range(1 << 6):
        bits = ramp + np.uint32(chunk * n)
        x = bits.view(np.float32)
        got = orc.cast(x, fmt)
        want = torch.from_numpy(x).to(tdt).view(torch.int16).numpy().view(np.uint16)
        if chunk in NAN_CHUNKS:
            nan_in = ((bits & 0x7f800000) == 0x7f800000) & ((bits & 0x007fffff) != 0)
            nan_out = ((got & exp_mask) == exp_mask) & ((got & man_mask) != 0)
            assert np.array_equal(nan_in, nan_out), chunk
            got[nan_in] = 0
            want = want.copy()
            want[nan_in] = 0
        if not np.array_equal(got, want):
            i = int(np.flatnonzero(got != want)[0])
            raise AssertionError(f"{fmt}: pattern {hex(int(bits[i]))} -> {hex(int(got[i]))}, torch {hex(int(want[i]))}")
