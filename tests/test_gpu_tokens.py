"""GPU parity of the 1 x 128 activation codec (wt_quantize_tokens) against
the CPU oracle, byte for byte on codes and bit for bit on scales: the flat
path (contiguous, hidden a multiple of 128), the strided vector path, the
element path, ragged last groups, and every (amax, element) pair of BF16
values."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import bf16_fp8_parameter_wt_b300 as wt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from bf16_fp8_parameter_wt_b300 import build
    build.build()
    assert torch.cuda.is_available()


def _tokens(tokens, hidden, seed, ld=None):
    """Seeded Student-t(3) x 0.02 BF16 activations with zero tokens, -0.0
    and +-3e4 outliers, as a (possibly strided) device tensor."""
    g = torch.Generator(device="cuda:0").manual_seed(seed)
    ld = ld or hidden
    z = torch.randn(tokens, ld, generator=g, device="cuda:0")
    chi = sum(torch.randn(tokens, ld, generator=g, device="cuda:0") ** 2 for _ in range(3))
    x = (z * 0.02 / torch.sqrt(chi / 3)).to(torch.bfloat16)
    if tokens > 2:
        x[1] = 0
        x[2, :min(ld, 9)] = -0.0
    if tokens * hidden > 1000:
        idx = torch.randint(0, tokens * hidden, (max(1, tokens // 4),), generator=g, device="cuda:0")
        xv = x[:, :hidden].reshape(-1) if ld == hidden else None
        if xv is not None:
            xv[idx] = 29952.0
    return x[:, :hidden]


def _oracle(oracle_mod, x):
    bits = x.cpu().view(torch.int16).numpy().view(np.uint16)
    return oracle_mod.quantize_tokens(bits)


def _run(x):
    tokens, hidden = x.shape
    codes = torch.full((tokens, hidden), 0xA5, dtype=torch.uint8, device="cuda:0")
    scales = torch.full((tokens, -(-hidden // 128)), -1.0, dtype=torch.float32, device="cuda:0")
    wt.wt_quantize_tokens(x.data_ptr(), tokens, hidden, x.stride(0), codes.data_ptr(),
                          scales.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("tokens,hidden,ld", [(4096, 7168, None), (128, 7168, None), (257, 7168, 7680),
                                              (5, 200, None), (3, 130, None), (7, 1000, 1003),
                                              (1, 1, None), (2, 128, None)])
def test_tokens_match_oracle(oracle_mod, tokens, hidden, ld):
    x = _tokens(tokens, hidden, 7 * tokens + hidden, ld)
    codes, scales = _run(x)
    want_c, want_s = _oracle(oracle_mod, x)
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))


def test_tokens_every_amax_element_pair(oracle_mod):
    """Each 1 x 128 group holds one amax a first, then BF16 values x with
    |x| <= a (both signs), padded with a; over all groups every pair of a
    positive finite BF16 amax and element appears."""
    rows = []
    per = 127
    for a in range(1, 0x7F80):
        vals = np.concatenate([np.arange(0, a + 1), np.arange(0x8000, 0x8000 + a + 1)])
        n = -(-vals.size // per)
        buf = np.full(n * per, a, dtype=np.int64)
        buf[:vals.size] = vals
        rows.append(np.concatenate([np.full((n, 1), a, np.int64), buf.reshape(n, per)],
                                   axis=1).astype(np.uint16))
    bits = np.concatenate(rows)
    del rows
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to("cuda:0")
    codes, scales = _run(x)
    del x
    n = max(1, len(os.sched_getaffinity(0)))
    chunks = np.array_split(np.arange(bits.shape[0]), n)
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda ix: oracle_mod.quantize_tokens(bits[ix[0]:ix[-1] + 1]), chunks))
    want_c = np.concatenate([p[0] for p in parts])
    want_s = np.concatenate([p[1] for p in parts])
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))


def test_tokens_refuses_misuse():
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device="cuda:0")
    codes = torch.empty(4, 256, dtype=torch.uint8, device="cuda:0")
    scales = torch.empty(4, 2, dtype=torch.float32, device="cuda:0")
    with pytest.raises(wt.WTError) as ei:
        wt.wt_quantize_tokens(x.data_ptr(), 4, 256, 128, codes.data_ptr(), scales.data_ptr())
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    with pytest.raises(wt.WTError) as ei:
        wt.wt_quantize_tokens(x.data_ptr(), 4, 256, 256, codes.data_ptr(), scales.data_ptr() + 2)
    assert ei.value.name == "WT_ERR_ALIGNMENT"
