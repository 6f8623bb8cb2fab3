"""GPU parity of the 1 x 128 activation codec (wt_quantize_tokens) against
the CPU oracle, byte for byte on codes and bit for bit on scales: the
shared-memory ring for large contiguous batches (stages from a ticket
counter or a fixed share per SM, many laps of the ring per CTA, ragged last
stages, the full dispatch batch the benchmark times, one ticket shared by
calls in stream order), the register kernel's flat, strided and element
paths, ragged last groups, and every (amax, element) pair of BF16 values; a
ring wait that gives up is reported by wt_tokens_check and the next call is
correct."""
import os
import time
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


def _run(x, ticket=None):
    tokens, hidden = x.shape
    codes = torch.full((tokens, hidden), 0xA5, dtype=torch.uint8, device="cuda:0")
    scales = torch.full((tokens, -(-hidden // 128)), -1.0, dtype=torch.float32, device="cuda:0")
    wt.wt_quantize_tokens(x.data_ptr(), tokens, hidden, x.stride(0), codes.data_ptr(),
                          scales.data_ptr(), torch.cuda.current_stream().cuda_stream,
                          ticket.data_ptr() if ticket is not None else 0)
    torch.cuda.synchronize()
    if ticket is not None:
        assert ticket.tolist() == [0, 0]          # every call leaves its counter zero
    return codes.cpu().numpy(), scales.cpu().numpy()


def _ticket():
    return torch.zeros(2, dtype=torch.int32, device="cuda:0")


# Batches of at least 16 (with a ticket counter) or 32 (without) stages of
# 128 groups per SM go through the shared-memory ring: 16384 x 7168 (48
# stages per SM: both), 8192 x 7168 (24: with a ticket), 700001 x 128 (37,
# last stage 97 groups: both), 300007 x 256 (32 - 0.3, last stage 78
# groups: with a ticket); strided rows of at least 32 groups too, one copy
# per row segment, always handed out per SM: 16384 x 7168 with rows 7296
# apart, 40001 x 4096 with rows 4104 apart (68 stages per SM, last stage 32
# groups). Smaller
# contiguous batches take the register kernel's flat path (4096 x 7168,
# 3001 x 7168, 128 x 7168, 1000 x 2048, 17 x 1024, 2 x 128), the rest its
# strided and element paths. Each case runs with and without a ticket.
@pytest.mark.parametrize("with_ticket", [False, True])
@pytest.mark.parametrize("tokens,hidden,ld", [(16384, 7168, None), (8192, 7168, None), (700001, 128, None),
                                              (300007, 256, None), (16384, 7168, 7296), (40001, 4096, 4104),
                                              (4096, 7168, None), (3001, 7168, None),
                                              (128, 7168, None), (1000, 2048, None), (17, 1024, None),
                                              (257, 7168, 7680), (5, 200, None), (3, 130, None),
                                              (7, 1000, 1003), (1, 1, None), (2, 128, None)])
def test_tokens_match_oracle(oracle_mod, tokens, hidden, ld, with_ticket):
    x = _tokens(tokens, hidden, 7 * tokens + hidden, ld)
    codes, scales = _run(x, _ticket() if with_ticket else None)
    want_c, want_s = _oracle(oracle_mod, x)
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))
    wt.wt_tokens_check()


def test_one_ticket_serves_calls_in_stream_order(oracle_mod):
    """Calls of different shapes share one ticket on one stream, back to
    back without a host wait: each equals the oracle."""
    xs = [_tokens(t, h, 31 * t + h) for t, h in [(8192, 7168), (700001, 128), (128, 7168), (8192, 7168)]]
    ticket = _ticket()
    outs = []
    for x in xs:
        t, h = x.shape
        c = torch.empty(t, h, dtype=torch.uint8, device="cuda:0")
        s_ = torch.empty(t, h // 128, dtype=torch.float32, device="cuda:0")
        wt.wt_quantize_tokens(x.data_ptr(), t, h, h, c.data_ptr(), s_.data_ptr(),
                              torch.cuda.current_stream().cuda_stream, ticket.data_ptr())
        outs.append((c, s_))
    wt.wt_tokens_check()
    assert ticket.tolist() == [0, 0]
    for x, (c, s_) in zip(xs, outs):
        want_c, want_s = _oracle(oracle_mod, x)
        assert np.array_equal(c.cpu().numpy(), want_c)
        assert np.array_equal(s_.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def _oracle_parallel(oracle_mod, bits):
    n = max(1, len(os.sched_getaffinity(0)))
    chunks = [c for c in np.array_split(np.arange(bits.shape[0]), n) if c.size]
    with ThreadPoolExecutor(len(chunks)) as ex:
        parts = list(ex.map(lambda ix: oracle_mod.quantize_tokens(bits[ix[0]:ix[-1] + 1]), chunks))
    return np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts])


def test_tokens_full_dispatch_batch(oracle_mod):
    """The batch the benchmark times (131072 tokens x 7168, launched the same
    way: through the ring, stages from a ticket counter), every code and
    scale against the oracle."""
    x = _tokens(131072, 7168, 1006)
    codes, scales = _run(x, _ticket())
    bits = x.cpu().view(torch.int16).numpy().view(np.uint16)
    del x
    want_c, want_s = _oracle_parallel(oracle_mod, bits)
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))
    wt.wt_tokens_check()


@pytest.mark.parametrize("with_ticket", [False, True])
def test_ring_wait_gives_up_then_recovers(oracle_mod, with_ticket):
    """One stage of a 16384 x 7168 batch is never copied (testing hook, 50 ms
    wait limit): the kernel returns by itself, wt_tokens_check reports
    WT_ERR_TIMEOUT once and clears it, the codes of the stalled stage are
    left unwritten, a ticket counter is left zero, and the next call is
    byte-exact."""
    x = _tokens(16384, 7168, 4242)
    want_c, want_s = _oracle(oracle_mod, x)
    ticket = _ticket() if with_ticket else None
    stalled = 1000 * 56 + 3                   # token 1000, group 3
    wt.wt_debug_tokens_stall_group(stalled, 50_000_000)
    try:
        t0 = time.perf_counter()
        codes, _ = _run(x, ticket)
        with pytest.raises(wt.WTError) as ei:
            wt.wt_tokens_check()
        assert ei.value.name == "WT_ERR_TIMEOUT"
        assert time.perf_counter() - t0 < 10.0
        assert (codes.reshape(-1, 128)[stalled] == 0xA5).all()
        wt.wt_tokens_check()                  # cleared
        # calls that do not use the ring ignore the hook
        xs = _tokens(64, 7168, 77, ld=7296)
        c2, s2 = _run(xs)
        w2 = _oracle(oracle_mod, xs)
        assert np.array_equal(c2, w2[0])
        wt.wt_tokens_check()
    finally:
        wt.wt_debug_tokens_stall_group(-1, 0)
    codes, scales = _run(x, ticket)
    wt.wt_tokens_check()
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
    want_c, want_s = _oracle_parallel(oracle_mod, bits)
    assert np.array_equal(codes, want_c)
    assert np.array_equal(scales.view(np.uint32), want_s.view(np.uint32))


def test_tokens_check_and_hook_refuse_misuse():
    with pytest.raises(wt.WTError) as ei:
        wt.wt_debug_tokens_stall_group(-2, 0)
    assert ei.value.name == "WT_ERR_INVALID_ARGUMENT"
    wt.wt_tokens_check()


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
