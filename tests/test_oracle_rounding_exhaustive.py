"""The oracle's float32 -> bf16 and float32 -> binary16 roundings on every
one of the 2^32 float32 bit patterns.

Both roundings decide every bf16 and fp16 result the GPU path is compared
with, so they are pinned in full rather than on a sample: against torch's
CPU casts (independent implementations of IEEE round-to-nearest-even), with
NaN inputs required to stay NaN (their payloads are not compared).  The
patterns are walked in 64 chunks of 2^26.
"""
import numpy as np
import torch

import oracle

CHUNK = 1 << 26


def _walk(convert_mine, torch_dtype, exp_mask, man_mask):
    base = np.arange(CHUNK, dtype=np.uint32)
    for k in range((1 << 32) // CHUNK):
        bits = base + np.uint32(k * CHUNK)
        f = bits.view(np.float32)
        mine = convert_mine(f)
        ref = torch.from_numpy(f).to(torch_dtype).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        if not nan.any():
            assert np.array_equal(mine, ref), f"chunk {k}"
            continue
        assert np.array_equal(mine[~nan], ref[~nan]), f"chunk {k}"
        m = mine[nan]
        assert np.all((m & exp_mask) == exp_mask) and np.all((m & man_mask) != 0), f"NaN lost in chunk {k}"


def test_bf16_rne_on_every_float32_pattern():
    _walk(oracle.bf16_rne, torch.bfloat16, 0x7F80, 0x007F)


def test_fp16_rne_on_every_float32_pattern():
    _walk(oracle.fp16_rne, torch.float16, 0x7C00, 0x03FF)
