"""Pins of the oracle's scale, element code, reassembly/fusion, layout and
coverage against library routines, exact-rational brute force, closed-form
sizes and invariants."""
import numpy as np
import pytest
import torch

import bruteforce as bf
from workloads import Output, Param, ValueRecipe, Workload, make_shards, shards_to_host_u16
from workloads import edge_stress, kimi_k2_moe_layer, llama_dense, llama_dense_tp4, tiny_dense, tp_slices_small


# --------------------------------------------------------------------------
# scale and element code
# --------------------------------------------------------------------------

def test_scale_matches_numpy_float32_division(oracle_mod):
    rng = np.random.default_rng(3)
    bits = np.concatenate([rng.integers(1, 0x7F7F, 200_000, dtype=np.uint32),
                           np.arange(1, 256, dtype=np.uint32)])     # bf16 subnormals
    amax = (bits << 16).astype(np.uint32).view(np.float32)
    want = amax / np.float32(448.0)                 # IEEE binary32 division
    got = np.array([oracle_mod.tile_scale(a) for a in amax[:20000]], np.float32)
    assert np.array_equal(got.view(np.uint32), want[:20000].view(np.uint32))
    assert oracle_mod.tile_scale(0.0) == np.float32(1.0)
    # subnormal scales do occur and stay exact
    tiny = np.float32(1e-40)
    assert oracle_mod.tile_scale(tiny) == tiny / np.float32(448.0)


def test_element_code_matches_exact_rational(oracle_mod):
    rng = np.random.default_rng(5)
    cases = []
    for _ in range(3000):
        a = int(rng.integers(1, 0x7F7F))
        x = int(rng.integers(0, a + 1)) | (int(rng.integers(0, 2)) << 15)
        cases.append((a, x))
    # adversarial: power-of-two scales (exact e4m3 ties), subnormal scales, x == amax
    for a in (0x43E0, 0x44E0, 0x3FE0, 0x0001, 0x0080, 0x0100, 0x2000, 0x7F7F):
        for x in (a, a - 1, 0x0000, 0x8000, a | 0x8000, 0x3F88, 0x3F98, 0x3FA8):
            if (x & 0x7FFF) <= a:
                cases.append((a, x))
    for a, x in cases:
        amax = bf.bf16_value(a)
        s_or = oracle_mod.tile_scale(float(amax))
        s_bf = bf.block_scale(amax)
        assert bf.Fraction(float(s_or)) == s_bf
        got = oracle_mod.quantize_element(x, s_or)
        want = bf.element_code(x, s_bf)
        assert got == want, (hex(a), hex(x), got, want)


def test_dequantisation_error_bound(oracle_mod):
    """|x - decode(q) * s| <= (ulp_e4m3(|y|)/2 + |y| 2^-24) * s, with the
    e4m3 ulp 2^-9 in the subnormal range and 2^(e-3) in binade e."""
    torch.manual_seed(0)
    w = Workload("bound", [Param("p", 512, 384, (100, 300, 112))],
                 [Output("o", (0,), True, (0,))], 1, ValueRecipe("student_t3", 0.02, 9))
    sh = make_shards(w)
    flat = shards_to_host_u16(sh)
    m = oracle_mod.Model(w)
    data, scales = m.prepare_output(0, flat)
    x = torch.cat(sh[0]).to(torch.float64).numpy()
    q = torch.from_numpy(data.reshape(512, 384).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.repeat(np.repeat(scales.reshape(4, 3).astype(np.float64), 128, 0), 128, 1)
    y = np.abs(x) / s
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    ulp = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    bound = (ulp / 2 + y * 2.0 ** -24) * s
    assert np.all(np.abs(x - q * s) <= bound * (1 + 1e-12))


# --------------------------------------------------------------------------
# reassembly, fusion, whole-output brute force
# --------------------------------------------------------------------------

def _tiny_cases():
    """Shapes with 1-4 uneven shards, fused and unfused, with zero blocks,
    -0.0, outliers and blocks whose scale is subnormal."""
    return [
        ("1x1", [Param("a", 1, 1, (1,))], [(0,)]),
        ("3x5", [Param("a", 3, 5, (2, 0, 1))], [(0,)]),
        ("128x128", [Param("a", 128, 128, (64, 64))], [(0,)]),
        ("256x1", [Param("a", 256, 1, (100, 100, 56))], [(0,)]),
        ("fused_129x130", [Param("a", 50, 130, (17, 33)), Param("b", 79, 130, (1, 0, 40, 38))],
         [(0, 1)]),
        ("three_parts", [Param("q", 64, 136, (32, 32)), Param("k", 32, 136, (32,)),
                         Param("v", 40, 136, (7, 33))], [(0, 1, 2)]),
    ]


def _fill_special(x: torch.Tensor, rng: np.random.Generator):
    """Plant zero blocks, -0.0, outliers and tiny magnitudes."""
    rows, cols = x.shape
    if rows * cols >= 4:
        x[0, 0] = -0.0
        x[-1, -1] = 0.0
    if rows >= 2 and cols >= 2:
        x[rows // 2, cols // 2] = 29952.0 * (1 if rng.integers(0, 2) else -1)
    if rows > 128 and cols >= 1:
        x[128:, :] = 0.0                      # an all-zero last block row
    return x


@pytest.mark.parametrize("case", range(len(_tiny_cases())))
def test_prepare_output_brute_force_tiny(oracle_mod, case):
    name, params, fusions = _tiny_cases()[case]
    rng = np.random.default_rng(100 + case)
    outputs = [Output(f"o{i}", f, True, (0,)) for i, f in enumerate(fusions)]
    w = Workload(name, params, outputs, 1, ValueRecipe("normal", 0.02, 50 + case))
    shards = make_shards(w)
    # plant specials in the reassembled tensors, then re-split
    for p, par in enumerate(params):
        full = _fill_special(torch.cat(shards[p]), rng)
        if case == 1:
            full.mul_(1e-38)                     # subnormal bf16 values -> subnormal scales
        r, new = 0, []
        for n in par.shard_rows:
            new.append(full[r:r + n].clone())
            r += n
        shards[p] = new
    flat = shards_to_host_u16(shards)
    m = oracle_mod.Model(w)
    for o, out in enumerate(outputs):
        fused = torch.cat([torch.cat(shards[p]) for p in out.parts])
        rows, cols = fused.shape
        bits = [int(v) & 0xFFFF for v in fused.view(torch.int16).flatten().tolist()]
        codes, scales = bf.quantize_matrix(bits, rows, cols)
        data, sc = m.prepare_output(o, flat)
        assert data.tolist() == codes
        assert [bf.Fraction(float(v)) for v in sc.tolist()] == scales


def test_bf16_passthrough_equals_torch_cat(oracle_mod):
    params = [Param("a", 37, 24, (10, 0, 27)), Param("b", 5, 24, (5,)), Param("n", 300, 1, (100, 100, 100))]
    outs = [Output("ab", (0, 1), False, (0,)), Output("n", (2,), False, (1,))]
    w = Workload("pt", params, outs, 2, ValueRecipe("normal", 1.0, 4))
    sh = make_shards(w)
    m = oracle_mod.Model(w)
    flat = shards_to_host_u16(sh)
    for o, out in enumerate(outs):
        want = torch.cat([torch.cat(sh[p]) for p in out.parts]).contiguous()
        got, _ = m.prepare_output(o, flat)
        assert got.tobytes() == want.view(torch.uint8).numpy().tobytes()


def test_fused_fp8_equals_quantised_torch_cat(oracle_mod):
    """Fusion then quantisation: the fused output equals the quantisation
    (numpy amax, numpy float32 division, torch e4m3 cast on the
    non-saturating range) of torch.cat of the reassembled parts."""
    params = [Param("w1", 256, 384, (64,) * 4), Param("w3", 256, 384, (100, 156, 0, 0))]
    w = Workload("fuse", params, [Output("gate_up", (0, 1), True, (0,))], 1,
                 ValueRecipe("normal", 0.006, 21))
    sh = make_shards(w)
    data, scales = oracle_mod.Model(w).prepare_output(0, shards_to_host_u16(sh))
    x = torch.cat([torch.cat(sh[0]), torch.cat(sh[1])]).float().numpy()
    blocks = x.reshape(4, 128, 3, 128).transpose(0, 2, 1, 3)
    amax = np.abs(blocks).max(axis=(2, 3)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1), amax / np.float32(448))
    assert np.array_equal(scales.reshape(4, 3), s)
    y = (blocks / s[:, :, None, None]).astype(np.float32)     # float32 / float32
    assert np.all(np.abs(y) <= 464)
    want = torch.from_numpy(y.transpose(0, 2, 1, 3).reshape(512, 384).copy())
    want = want.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(data.reshape(512, 384), want)


# --------------------------------------------------------------------------
# layout and coverage
# --------------------------------------------------------------------------

def _ranges(w, d, s):
    out = []
    for o, outp in enumerate(w.outputs):
        m, n = w.output_shape(o)
        db = m * n * (1 if outp.fp8 else 2)
        sb = 4 * (-(-m // 128)) * (-(-n // 128)) if outp.fp8 else 0
        for k, r in enumerate(outp.dst_ranks):
            out.append((r, d[o][k], db))
            if outp.fp8:
                out.append((r, s[o][k], sb))
    return out


@pytest.mark.parametrize("make", [tiny_dense, llama_dense, kimi_k2_moe_layer, edge_stress])
def test_layout_disjoint_aligned_and_tight(oracle_mod, make):
    w = make()
    d, s, pools = oracle_mod.Model(w).layout()
    rs = _ranges(w, d, s)
    for rank in range(w.num_ranks):
        mine = sorted((off, n) for r, off, n in rs if r == rank)
        end = 0
        for off, n in mine:
            assert off % 256 == 0 and off >= end
            assert off - end < 256                      # no gap beyond alignment
            end = off + n
        assert pools[rank] == (-(-end // 256)) * 256


def test_layout_closed_form_pool_sizes(oracle_mod):
    # Kimi-K2-shaped layer: per expert gate_up 4096x7168 codes + 32x56 scales,
    # down 7168x2048 codes + 56x16 scales, all multiples of 256 bytes;
    # rank 0 holds experts 0, 8, ..., 384 (49), ranks 1..7 hold 48.
    per_expert = 4096 * 7168 + 32 * 56 * 4 + 7168 * 2048 + 56 * 16 * 4
    assert per_expert == 44_050_944
    _, _, pools = oracle_mod.Model(kimi_k2_moe_layer()).layout()
    assert pools == [49 * per_expert] + [48 * per_expert] * 7
    assert sum(pools) == 16_959_613_440
    # edge set: ranks 3 and 4 receive nothing; rank 1's 1000x7168 codes are
    # followed by ceil(1000/128) x 56 scales at the next 256-byte boundary
    _, _, pools = oracle_mod.Model(edge_stress()).layout()
    assert pools[3] == 0 and pools[4] == 0
    assert pools[1] == 1000 * 7168 + 8 * 56 * 4
    # rank 0: 7168x2050 codes (14694400 = 57400 x 256) + 56x17 scales (3808 bytes),
    # the pool end rounded up to 256
    assert pools[0] == 14_694_400 + 3808 + 32
    assert pools[2] == 163840 * 7168 * 2


def test_layout_explicit_offsets_and_replicas(oracle_mod):
    params = [Param("a", 128, 256, (128,)), Param("b", 64, 64, (64,))]
    outs = [Output("a", (0,), True, (0, 1), data_off=(4096, None), scale_off=(0, None)),
            Output("b", (1,), False, (0, 0))]
    w = Workload("explicit", params, outs, 2)
    d, s, pools = oracle_mod.Model(w).layout()
    assert d[0] == [4096, 0] and s[0][0] == 0
    assert s[0][1] == 128 * 256                 # after the auto data on rank 1
    # auto ranges on rank 0 start after the explicit end 4096 + 32768
    assert d[1] == [4096 + 32768, 4096 + 32768 + 8192]
    assert pools == [4096 + 32768 + 2 * 8192, 128 * 256 + 256]


def test_prepare_covers_every_scheduled_byte_once(oracle_mod):
    """Two runs into pools pre-filled with different canaries: scheduled
    bytes agree (so each was written), padding keeps its canary."""
    w = tiny_dense()
    sh = shards_to_host_u16(make_shards(w))
    m = oracle_mod.Model(w)
    d, s, pools = m.layout()
    a = m.prepare(sh, nthreads=3, fill=0x00)
    b = m.prepare(sh, nthreads=1, fill=0xFF)
    for rank in range(w.num_ranks):
        mask = np.zeros(pools[rank], bool)
        for r, off, n in _ranges(w, d, s):
            if r == rank:
                assert not mask[off:off + n].any()
                mask[off:off + n] = True
        assert np.array_equal(a[rank][mask], b[rank][mask])
        assert np.all(a[rank][~mask] == 0x00) and np.all(b[rank][~mask] == 0xFF)


# --------------------------------------------------------------------------
# tensor-parallel destination slices
# --------------------------------------------------------------------------

def _expected_slice(data, scales, shape, sl, fp8):
    """numpy slicing of a whole prepared output (codes and block scales)."""
    m, n = shape
    es = 1 if fp8 else 2
    arr = data.reshape(m, n * es)
    grid = scales.reshape(-(-m // 128), -(-n // 128)) if fp8 else None
    if sl is None:
        return arr.ravel(), (grid.ravel() if fp8 else None)
    dim, ranges = sl
    if dim == 0:
        d = np.concatenate([arr[b:b + k] for b, k in ranges])
        g = np.concatenate([grid[b // 128:-(-(b + k) // 128)] for b, k in ranges]) if fp8 else None
    else:
        d = np.concatenate([arr[:, b * es:(b + k) * es] for b, k in ranges], axis=1)
        g = (np.concatenate([grid[:, b // 128:-(-(b + k) // 128)] for b, k in ranges], axis=1)
             if fp8 else None)
    return d.ravel(), (g.ravel() if fp8 else None)


def test_slices_equal_numpy_slicing_of_the_whole_output(oracle_mod):
    w = tp_slices_small()
    flat = shards_to_host_u16(make_shards(w))
    m = oracle_mod.Model(w)
    pools = m.prepare(flat, nthreads=2)
    d_off, s_off, _ = m.layout()
    for o, out in enumerate(w.outputs):
        data, scales = m.prepare_output(o, flat)
        for d, rank in enumerate(out.dst_ranks):
            sl = out.slices[d]
            want_d, want_s = _expected_slice(data, scales, w.output_shape(o), sl, out.fp8)
            assert m.dst_shape(o, d) == w.dst_shape(o, d)
            got_d = pools[rank][d_off[o][d]:d_off[o][d] + want_d.size]
            assert np.array_equal(got_d, want_d), (out.name, d)
            if out.fp8:
                got_s = pools[rank][s_off[o][d]:s_off[o][d] + 4 * want_s.size].view(np.float32)
                assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), (out.name, d)


def test_tensor_parallel_slices_reassemble_the_tensor(oracle_mod):
    """Row slices that partition the fused tensor, concatenated in range
    order, are the whole output; so are column slices side by side."""
    params = [Param("g", 512, 384, (128,) * 4), Param("u", 512, 384, (256, 256)),
              Param("g2", 512, 384, (512,)), Param("u2", 512, 384, (512,))]
    tp = 2
    rows = [(0, ((r * 256, 256), (512 + r * 256, 256))) for r in range(tp)]   # gate_r, up_r
    cols = [(1, ((c * 128, 128),)) for c in range(3)]
    outs = [Output("gu", (0, 1), True, tuple(range(tp)), slices=tuple(rows)),
            Output("gu_cols", (2, 3), True, (0, 1, 0), slices=tuple(cols))]
    w = Workload("tp", params, outs, tp, ValueRecipe("normal", 0.02, 43))
    flat = shards_to_host_u16(make_shards(w))
    m = oracle_mod.Model(w)
    pools = m.prepare(flat, nthreads=2)
    d_off, s_off, _ = m.layout()
    data, scales = m.prepare_output(0, flat)
    whole = data.reshape(1024, 384)
    grid = scales.reshape(8, 3)
    pieces, gpieces = {}, {}
    for r in range(tp):
        blob = pools[r][d_off[0][r]:d_off[0][r] + 512 * 384].reshape(512, 384)
        sb = pools[r][s_off[0][r]:s_off[0][r] + 4 * 4 * 3].view(np.float32).reshape(4, 3)
        pieces[r * 256], pieces[512 + r * 256] = blob[:256], blob[256:]
        gpieces[r * 2], gpieces[4 + r * 2] = sb[:2], sb[2:]
    assert np.array_equal(np.concatenate([pieces[k] for k in sorted(pieces)]), whole)
    assert np.array_equal(np.concatenate([gpieces[k] for k in sorted(gpieces)]).view(np.uint32),
                          grid.view(np.uint32))
    data2, scales2 = m.prepare_output(1, flat)
    cols_got = [pools[out_rank][d_off[1][d]:d_off[1][d] + 1024 * 128].reshape(1024, 128)
                for d, out_rank in enumerate(outs[1].dst_ranks)]
    assert np.array_equal(np.concatenate(cols_got, axis=1), data2.reshape(1024, 384))


@pytest.mark.parametrize("sl", [(0, ((64, 128),)), (0, ((0, 100), (128, 128))), (0, ((0, 256), (128, 128))),
                                (0, ((256, 128),)), (1, ((0, 200),)), (2, ((0, 128),)), (0, ((0, 0),))])
def test_invalid_slices_are_rejected(oracle_mod, sl):
    w = Workload("bad", [Param("p", 300, 260, (300,))],
                 [Output("p", (0,), True, (0,), slices=(sl,))], 1)
    with pytest.raises(ValueError):
        oracle_mod.Model(w).layout()


# --------------------------------------------------------------------------
# completion counts per rank
# --------------------------------------------------------------------------

def test_expected_blocks_closed_forms(oracle_mod):
    w = kimi_k2_moe_layer()
    m = oracle_mod.Model(w)
    per_expert = (4096 // 128) * (7168 // 128) + (7168 // 128) * (2048 // 128)   # 2688
    assert [m.expected_blocks(r) for r in range(8)] == [49 * per_expert] + [48 * per_expert] * 7
    tp = llama_dense_tp4()
    mt = oracle_mod.Model(tp)
    counts = [mt.expected_blocks(r) for r in range(4)]
    whole = llama_dense()
    blocks = whole.num_tiles
    norm_blocks = sum(32 for o in whole.outputs if o.name.endswith("norm"))   # [4096, 1]: 32 x 1
    assert sum(counts) == blocks + 3 * norm_blocks      # the norms go to all four ranks
    # ranks differ only in their vocabulary rows of the embedding and lm_head
    assert counts[0] == counts[1] == counts[2]
    assert counts[0] - counts[3] == (32128 - 31872) // 128 * 32 * 2
    ts = tp_slices_small()
    ms = oracle_mod.Model(ts)
    # rank 0: 'a' whole (3x3), 'a' rows 256..300 (1x3), 'a' cols [0,128)+[256,260) (3x2); 'b' rows (2x2)
    assert ms.expected_blocks(0) == 9 + 3 + 6 + 4
    # rank 1: 'a' rows (2x3), 'a' cols [128,260) (3x2); 'b' whole (2x2) and cols [128,136) (2x1)
    assert ms.expected_blocks(1) == 6 + 6 + 4 + 2
