"""The e4m3 convert that every code of the library goes through, against the
CPU definition of the format (the oracle's E, written from the format's
definition) on every one of the 2^32 fp32 bit patterns: round to nearest
even, saturation to +-448 (also of +-inf), signed zeros and subnormal codes.
NaN inputs only have to give a NaN code (0x7F or 0xFF): the product path
never sees one."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt
from gpu_helpers import ncores

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def test_gpu_convert_equals_the_format_definition_on_every_fp32(oracle_mod):
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    sub = CHUNK // 16
    with ThreadPoolExecutor(ncores()) as ex:
        for first in range(0, 1 << 32, CHUNK):
            wt.wt_debug_e4m3_encode(first, CHUNK, out.data_ptr(), stream)
            want = np.concatenate(list(ex.map(lambda k: oracle_mod.e4m3_encode_bits_range(first + k * sub, sub),
                                              range(16))))
            got = out.cpu().numpy()
            bits = np.arange(first, first + CHUNK, dtype=np.uint64).astype(np.uint32)
            nan = ((bits >> 23) & 0xFF == 0xFF) & ((bits & 0x7FFFFF) != 0)
            bad = (got != want) & ~nan
            if bad.any():
                i = int(np.nonzero(bad)[0][0])
                raise AssertionError(f"fp32 0x{int(bits[i]):08x}: gpu 0x{got[i]:02x}, definition 0x{want[i]:02x}")
            assert np.all((got[nan] & 0x7F) == 0x7F)


def test_sweep_hook_refuses_ranges_past_the_last_pattern():
    with pytest.raises(wt.WTError) as ei:
        wt.wt_debug_e4m3_encode(0xFFFFFFFF, 2, 1, 0)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
