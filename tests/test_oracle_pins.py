"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages fix or a hand-derived worked example (tests/golden), a library routine
(torch's bf16 / float8_e4m3fn conversions, numpy cos/sin), a closed form, an
invariant, or brute force on tiny inputs.  The sources are
metrale_model_arch/deepseek_v41_ref/compress.rs (the CPU reference) and
metrale_model_arch/attn_v41/forward.rs (AttnV41::forward).
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]


def _structured_f32(seed=0):
    """Every exponent/top-mantissa pattern (upper 16 bits) combined with the
    low half-words that decide a rounding: 0, 1, 0x7fff, 0x8000, 0x8001,
    0xffff and two random ones.  NaNs are dropped."""
    rng = np.random.default_rng(seed)
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF], np.uint32)
    lows = np.concatenate([lows, rng.integers(0, 1 << 16, 2).astype(np.uint32)])
    u = (hi[:, None] | lows[None, :]).ravel()
    x = u.view(np.float32)
    return x[~np.isnan(x)]


# ---------------------------------------------------------------------------
# Pin 1: scalar codecs
# ---------------------------------------------------------------------------
def _e2m1_by_midpoints(x):
    """Independent e2m1 rounding: compare |x| against the seven midpoints,
    closed on the side of the even code (compress.rs to_e2m1_rne's tie rule)."""
    a = np.abs(x.astype(np.float64))
    out = np.select(
        [a <= 0.25, a < 0.75, a <= 1.25, a < 1.75, a <= 2.5, a < 3.5, a <= 5.0],
        [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0], 6.0)
    return np.copysign(out, x).astype(np.float32)


def test_e2m1_golden_ties(orc):
    for ln in _golden_lines("e2m1_ties.txt"):
        x, want, clamp = ln.split()
        v = np.float32(float(x))
        if int(clamp):
            v = np.float32(np.clip(v, -6, 6))
        got = orc.to_e2m1(np.array([v], np.float32))[0]
        w = np.float32(float(want))
        assert got == w and np.signbit(got) == np.signbit(w), (x, got, want)


def test_e2m1_sweep_against_midpoints(orc):
    x = _structured_f32()
    x = x[np.abs(x) <= 8.0]
    extra = []
    for mid in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0):
        m = np.float32(mid)
        for k in range(-3, 4):
            extra.append(np.nextafter(m, np.float32(np.inf if k > 0 else -np.inf))
                         if k else m)
    x = np.concatenate([x, np.array(extra, np.float32), -np.array(extra, np.float32)])
    got = orc.to_e2m1(x)
    want = _e2m1_by_midpoints(x)
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))


def test_bf16_rne_against_torch(orc):
    x = _structured_f32(1)
    x = x[np.isfinite(x) | np.isinf(x)]
    got = orc.f32_to_bf16(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # torch's conversion is a library RNE; NaNs were dropped above.
    assert np.array_equal(got, want)


def _e4m3_table():
    """All 256 e4m3 codes decoded by torch's float8_e4m3fn (library routine)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def test_e4m3_decode_against_torch(orc):
    table = _e4m3_table()
    got = orc.e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    nan = np.isnan(table)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], table[~nan])


def _e4m3_brute(x):
    """Nearest finite e4m3 value by brute force over all codes, ties to the even
    code, saturating (448 is the largest finite value)."""
    table = _e4m3_table()
    pos = np.arange(128)
    pos = pos[~np.isnan(table[pos])]
    vals = table[pos]
    out = np.empty(x.shape, np.uint8)
    for i, v in enumerate(x.astype(np.float64)):
        a = abs(v)
        d = np.abs(vals - a)
        best = np.flatnonzero(d == d.min())
        if best.size > 1:
            best = best[(pos[best] % 2) == 0]
        c = int(pos[best[0]])
        out[i] = c | (0x80 if np.signbit(v) else 0)
    return out


def test_e4m3_encode_against_brute_force(orc):
    table = _e4m3_table()
    fin = np.sort(np.unique(np.abs(table[~np.isnan(table)])))
    mids = (fin[:-1] + fin[1:]) / 2  # exact in f32: neighbours differ by a power of two
    rng = np.random.default_rng(2)
    xs = [fin, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
          np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
          rng.uniform(0, 500, 2000), np.exp2(rng.uniform(-14, 9, 2000)),
          np.array([0.0, 448.0, 463.9, 464.0, 470.0, 1e6, 1e-12])]
    x = np.concatenate([np.asarray(v, np.float64) for v in xs]).astype(np.float32)
    x = np.concatenate([x, -x])
    got = orc.f32_to_e4m3(x)
    want = _e4m3_brute(x)
    assert np.array_equal(got, want)
    # In range, torch's own (library) conversion must agree as well.
    inr = np.abs(x) <= 448
    tv = torch.from_numpy(x[inr].copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[inr], tv)


def test_pow2_ceil_properties(orc):
    rng = np.random.default_rng(3)
    x = np.concatenate([np.exp2(rng.uniform(-126, 127, 5000)),
                        np.exp2(np.arange(-126, 127).astype(np.float64)),
                        np.exp2(np.arange(-126, 127).astype(np.float64)) * 1.0000001]
                       ).astype(np.float32)
    x = x[np.isfinite(x) & (x > 0)]
    got = orc.pow2_ceil(x).astype(np.float64)
    xd = x.astype(np.float64)
    mant, _ = np.frexp(got)
    assert np.all(mant == 0.5)                # a power of two
    assert np.all(got >= xd)                  # not below x
    assert np.all(got / 2 < xd)               # the smallest such power


# ---------------------------------------------------------------------------
# Pins 2-3: block quantisers
# ---------------------------------------------------------------------------
def _bf16_bits_of(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_fp4_quant_golden_examples(orc):
    for ln in _golden_lines("fp4_quant_examples.txt"):
        name, mode, block, sbyte, ins, outs = [p.strip() for p in ln.split("|")]
        block = int(block)
        xin = np.zeros(block, np.float32)
        v = [float(s) for s in ins.split()]
        xin[:len(v)] = v
        want = np.zeros(block, np.float32)
        w = [float(s) for s in outs.split()]
        want[:len(w)] = w
        y, codes, scales = orc.fp4_quant(_bf16_bits_of(xin)[None, :], block, mode == "e4m3")
        got = orc.bf16_to_f32(y[0])
        assert np.array_equal(got, want), (name, got[:8], want[:8])
        assert np.array_equal(np.signbit(got), np.signbit(want)), name
        assert int(scales[0, 0]) == int(sbyte), (name, scales[0, 0])


def _nearest_on_grid_ok(x, y, s):
    """Brute force: y/s is a grid point and no grid point is nearer to the
    clamped x/s; on equal distance y/s must carry the even code."""
    t = np.clip(x.astype(np.float64) / s, -6, 6)
    g = y.astype(np.float64) / s
    a = np.abs(t)
    d = np.abs(GRID[None, :] - a[:, None])
    dmin = d.min(axis=1)
    idx = np.abs(GRID[None, :] - np.abs(g)[:, None]).argmin(axis=1)
    on_grid = np.isin(np.abs(g), GRID)
    nearest = np.isclose(d[np.arange(len(a)), idx], dmin, rtol=0, atol=0)
    tie = (d == dmin[:, None]).sum(axis=1) > 1
    even_ok = ~tie | (idx % 2 == 0)
    return on_grid & nearest & even_ok


@pytest.mark.parametrize("e4m3,block", [(False, 32), (True, 16)])
def test_fp4_quant_properties(orc, e4m3, block):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 20
    x[3] = 0.0                      # zero row: floors
    x[5, :block] = 6 * 2.0 ** 3     # amax exactly 6*2^k
    xb = _bf16_bits_of(x)
    y, codes, scales = orc.fp4_quant(xb, block, e4m3)
    xf = orc.bf16_to_f32(xb).reshape(64, -1, block).astype(np.float64)
    yf = orc.bf16_to_f32(y).reshape(64, -1, block).astype(np.float64)
    amax = np.maximum(np.abs(xf).max(axis=2),
                      6 * 2.0 ** (-9 if e4m3 else -126))
    table = _e4m3_table()
    for r in range(64):
        for b in range(xf.shape[1]):
            if e4m3:
                s = table[scales[r, b]]
                # the scale is the e4m3 value nearest amax/6 (brute force)
                fin = table[:127]
                near = np.abs(fin - amax[r, b] / 6)
                assert near[scales[r, b]] == near.min()
            else:
                s = 2.0 ** (int(scales[r, b]) - 127)
                assert amax[r, b] / 6 <= s < 2 * amax[r, b] / 6
            ok = _nearest_on_grid_ok(xf[r, b], yf[r, b], s)
            assert ok.all(), (r, b)
            # the sign survives, zeros included
            assert np.array_equal(np.signbit(yf[r, b]) | (yf[r, b] == 0),
                                  np.signbit(xf[r, b]) | (yf[r, b] == 0))
    # codes: low nibble = even element, value = grid[idx] * s with the sign bit
    c = np.stack([codes & 15, codes >> 4], axis=-1).reshape(64, -1, block)
    sgn = np.where(c & 8, -1.0, 1.0)
    mag = GRID[c & 7]
    if e4m3:
        s_all = table[scales][:, :, None]
    else:
        s_all = (2.0 ** (scales.astype(np.int64) - 127))[:, :, None]
    assert np.array_equal(sgn * mag * s_all, yf)
    # floors: zero row -> smallest scale, zero outputs
    assert np.all(scales[3] == 1) and np.all(yf[3] == 0)
    if not e4m3:
        assert scales[5, 0] == 127 + 3


def test_e8m0_quant_idempotent(orc):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((128, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.02] *= 20
    y1, _, _ = orc.fp4_quant(_bf16_bits_of(x), 32, False)
    y2, _, _ = orc.fp4_quant(y1, 32, False)
    assert np.array_equal(y1, y2)


# ---------------------------------------------------------------------------
# Pin 4: YaRN table and rotary
# ---------------------------------------------------------------------------
def test_yarn_factor_one_is_plain_rope(orc):
    f = orc.yarn_inv_freqs(64, 65536, 160000.0, 1.0, 32.0, 1.0).astype(np.float64)
    i = np.arange(32)
    want = 160000.0 ** (-(2 * i) / 64)
    assert np.allclose(f, want, rtol=3e-7, atol=0)


def test_yarn_ramp_closed_form(orc):
    # Hand-computed bounds for dim 64, original length 65536, base 160000:
    # corr(32) = 15.45 -> low 15, corr(1) = 24.71 -> high 25 (see
    # tests/golden/yarn_bounds.txt).
    low, high = 15, 25
    factor = 16.0
    f = orc.yarn_inv_freqs(64, 65536, 160000.0, factor, 32.0, 1.0).astype(np.float64)
    i = np.arange(32)
    base = 160000.0 ** (-(2 * i) / 64)
    ramp = np.clip((i - low) / (high - low), 0, 1)
    want = base * (1 - ramp) + base / factor * ramp
    assert np.allclose(f, want, rtol=1e-6, atol=0)
    assert np.allclose(f[: low + 1], base[: low + 1], rtol=3e-7)
    assert np.allclose(f[high:], base[high:] / factor, rtol=3e-7)


def test_yarn_table_values(orc):
    fc = orc.yarn_freqs_cis(64, 3000)
    f = orc.yarn_inv_freqs(64, 65536, 160000.0, 16.0, 32.0, 1.0)
    assert np.all(fc[0, :, 0] == 1.0) and np.all(fc[0, :, 1] == 0.0)
    p = np.arange(3000, dtype=np.float32)[:, None]
    ang = (p * f[None, :]).astype(np.float32).astype(np.float64)  # one f32 product
    assert np.allclose(fc[..., 0], np.cos(ang), rtol=0, atol=3e-7)
    assert np.allclose(fc[..., 1], np.sin(ang), rtol=0, atol=3e-7)
    assert np.allclose(fc[..., 0].astype(np.float64) ** 2 + fc[..., 1].astype(np.float64) ** 2,
                       1.0, atol=1e-6)


def test_rotary_dims_pairs_and_sign(orc):
    hd, rd = 12, 4
    # a table with two positions: angle 90 degrees exactly (c=0, s=1) for both columns
    fc = np.zeros((2, rd // 2, 2), np.float32)
    fc[0, :, 0] = 1.0
    fc[1, :, 1] = 1.0
    x = np.arange(1, hd + 1, dtype=np.float32)[None, :]
    y = orc.apply_rotary(x, rd, [1], fc)
    assert np.array_equal(y[0, : hd - rd], x[0, : hd - rd])          # nope dims untouched
    x0, x1, x2, x3 = x[0, hd - rd:]
    assert list(y[0, hd - rd:]) == [-x1, x0, -x3, x2]                  # (x0,x1) -> (-x1, x0)
    yi = orc.apply_rotary(y, rd, [1], fc, inverse=True)
    assert np.array_equal(yi, x)
    y0 = orc.apply_rotary(x, rd, [0], fc)
    assert np.array_equal(y0, x)


def test_rotary_preserves_pair_norms(orc):
    rng = np.random.default_rng(6)
    fc = orc.yarn_freqs_cis(16, 100)
    x = rng.standard_normal((50, 64)).astype(np.float32)
    pos = rng.integers(0, 100, 50)
    y = orc.apply_rotary(x, 16, pos, fc)
    n0 = (x[:, 48:].reshape(50, 8, 2).astype(np.float64) ** 2).sum(-1)
    n1 = (y[:, 48:].reshape(50, 8, 2).astype(np.float64) ** 2).sum(-1)
    assert np.allclose(n0, n1, rtol=1e-5)
    back = orc.apply_rotary(y, 16, pos, fc, inverse=True)
    assert np.allclose(back, x, atol=1e-5)


# ---------------------------------------------------------------------------
# Pin 5: window ring and window indices
# ---------------------------------------------------------------------------
def _pos_rows(positions, hd=4):
    """Rows whose every element encodes a position (bf16-exact integers < 256
    are not enough, so split the position over two elements)."""
    p = np.asarray(positions, np.int64)
    rows = np.zeros((len(p), hd), np.float32)
    rows[:, 0] = p // 128
    rows[:, 1] = p % 128
    rows[:, 2] = 1.0  # marks a written row
    return _bf16_bits_of(rows)


def _decode_pos(rows_bits):
    f = np.asarray(rows_bits).view(np.uint16).astype(np.uint32) << 16
    v = f.view(np.float32)
    return (v[:, 0].astype(np.int64) * 128 + v[:, 1].astype(np.int64),
            v[:, 2] == 1.0)


def test_ring_golden(orc):
    for ln in _golden_lines("ring_examples.txt"):
        lhs, rhs = ln.split("|")
        win, m, sp = map(int, lhs.split())
        want = rhs.split()
        ring0 = np.zeros((win, 4), np.uint16)
        kv = _pos_rows(range(sp, sp + m))
        ring, _ = orc.window_ring_write(kv, ring0, win, sp)
        pos, written = _decode_pos(ring)
        got = [str(p) if w else "-" for p, w in zip(pos, written)]
        assert got == want, (ln, got)


def _page_split_ring(kv_pos, win, start_pos, ring_pos):
    """The printed copies of forward.rs, restated: whole rows at start_pos 0
    (split at cutoff = m mod win when m > win), one row at slot start_pos mod
    win otherwise.  Positions stand for rows."""
    ring = list(ring_pos)
    m = len(kv_pos)
    if start_pos == 0:
        if m <= win:
            ring[:m] = kv_pos
        else:
            cutoff = m % win
            tail = kv_pos[m - win:]
            ring[cutoff:win] = tail[: win - cutoff]
            ring[:cutoff] = tail[win - cutoff:]
    else:
        ring[start_pos % win] = kv_pos[0]
    return ring


def test_ring_matches_printed_copies_bruteforce(orc):
    """The oracle's ring (newest row per slot) against the page's own copy
    pattern, for every win < 13, m < 30 at position 0 and every decode
    position < 30."""
    for win in range(1, 13):
        for m in range(1, 30):
            for sp in [0] + list(range(1, 30)):
                if sp > 0 and m > 1:
                    continue  # the printed copies cover m == 1 past position 0
                before = [1000 + j for j in range(win)]
                ring0 = _pos_rows(before)
                kv = _pos_rows(range(sp, sp + m))
                ring, _ = orc.window_ring_write(kv, ring0, win, sp)
                got = list(_decode_pos(ring)[0])
                want = _page_split_ring(list(range(sp, sp + m)), win, sp, before)
                assert got == want, (win, m, sp, got, want)


def test_window_indices_see_exactly_their_window(orc):
    """Every (win, m, start_pos) up to 40: the rows the window indices of a
    query point at hold exactly the positions max(0, p-win+1) .. p."""
    for win in (1, 2, 3, 5, 8, 16, 40):
        for m in (1, 2, 3, 7, 16, 39, 40):
            for sp in (0, 1, 2, 5, 17, 39, 40, 100):
                kv = _pos_rows(range(sp, sp + m))
                # the ring before the call holds positions sp-win .. sp-1 at q mod win
                ring_pos = np.full(win, -1, np.int64)
                for q in range(sp - win, sp):
                    if q >= 0:
                        ring_pos[q % win] = q
                ring0 = _pos_rows(np.where(ring_pos < 0, 0, ring_pos))
                ring0_f = ring0.copy()
                ring0_f[ring_pos < 0, 2] = 0  # unwritten slots carry no mark
                _, rows_a = orc.window_ring_write(kv, ring0_f, win, sp)
                assert rows_a.shape[0] == orc.rows_a_len(m, win, sp)
                idx = orc.window_topk_idxs(win, m, sp)
                apos, awritten = _decode_pos(rows_a)
                for t in range(m):
                    p = sp + t
                    valid = idx[t][idx[t] >= 0]
                    assert np.all(valid < rows_a.shape[0])
                    assert np.all(awritten[valid])
                    got = sorted(apos[valid].tolist())
                    assert got == list(range(max(0, p - win + 1), p + 1)), (win, m, sp, t)
                    assert (idx[t] < 0).sum() == max(0, win - (p + 1))


# ---------------------------------------------------------------------------
# Latent write: positions and cache placement (forward.rs latent branch)
# ---------------------------------------------------------------------------
def test_latent_write_positions_and_rows(orc):
    hd, rd, ratio = 32, 8, 4
    fc = orc.yarn_freqs_cis(rd, 200)
    rng = np.random.default_rng(7)
    for sp, m in [(0, 16), (0, 19), (11, 1), (15, 1), (35, 20)]:
        G = orc.new_groups(m, ratio, sp)
        lat = _bf16_bits_of(rng.standard_normal((max(G, 0), hd)).astype(np.float32))
        cache0 = _bf16_bits_of(np.full((60, hd), 7.0, np.float32))
        cache, codes, scales = orc.compress_latent_write(lat, fc, cache0, rd, ratio, sp, m)
        first = sp // ratio
        changed = np.flatnonzero((cache != cache0).any(axis=1))
        assert set(changed.tolist()) <= set(range(first, first + G))
        if sp > 0 and m == 1:
            # the one decode group exists only when sp+1 is a multiple of ratio,
            # and its rope position is sp + 1 - ratio
            assert G == (1 if (sp + 1) % ratio == 0 else 0)
        for g in range(G):
            lpos = (first + g) * ratio
            if sp > 0 and m == 1:
                assert lpos == sp + 1 - ratio
            row = orc.bf16_to_f32(lat[g])[None, :]
            rot = orc.apply_rotary(row, rd, [lpos], fc)
            rb = orc.f32_to_bf16(rot)
            want, _, _ = orc.fp4_quant(rb, 16, True)
            assert np.array_equal(cache[first + g], want[0])


def _groups_by_enumeration(m, ratio, sp):
    """Walk the positions one by one: position p completes a group of
    ``ratio`` consecutive positions when it is the group's last one
    ((p + 1) % ratio == 0).  Returns (groups complete after the call, groups
    completed by this call)."""
    total = new = 0
    for p in range(sp + m):
        if (p + 1) % ratio == 0:
            total += 1
            if p >= sp:
                new += 1
    return total, new


def test_group_counts_by_enumeration(orc):
    """compress_len (forward.rs / compress.rs: compressed rows that exist after
    the call) and the groups a call completes, against a walk over every
    position; plus the row the latent copy starts at (start_pos / ratio =
    groups complete before the call) and the latent write's own count."""
    for ratio in (1, 2, 3, 4, 7, 16, 128):
        for sp in sorted({0, 1, 2, 3, ratio - 1, ratio, ratio + 1, 37, 255, 256, 300}):
            for m in (1, 2, 3, 4, 5, 8, 13, 64, 129, 300):
                total, new = _groups_by_enumeration(m, ratio, sp)
                assert orc.compress_len(m, ratio, sp) == total, (m, ratio, sp)
                assert orc.new_groups(m, ratio, sp) == new, (m, ratio, sp)
                before, _ = _groups_by_enumeration(sp, ratio, 0) if sp > 0 else (0, 0)
                assert total - new == before
    # the latent write takes exactly its own count of rows
    fc = orc.yarn_freqs_cis(8, 64)
    lat = np.zeros((2, 32), np.uint16)
    with pytest.raises(AssertionError):
        orc.compress_latent_write(lat, fc, np.zeros((16, 32), np.uint16), 8, 4, 0, 4)


def test_merged_row_length(orc):
    """The merged index row (forward.rs / compress.rs merge: the window indices,
    then the indexer's ctopk picks, none while no compressed row exists)."""
    for win in (1, 16, 128):
        for topk in (1, 8, 512, 2048):
            for n_c in (0, 1, 7, 512, 520, 32768):
                want = win + (0 if n_c == 0 else min(topk, n_c))
                assert orc.merged_len(win, topk, n_c) == want


def test_attn_scale(orc):
    """compress.rs attention_any: scale = head_dim^-0.5 in f32."""
    assert orc.attn_scale(64) == 0.125 and orc.attn_scale(256) == 0.0625
    for hd in (128, 512):
        exact = hd ** -0.5
        got = orc.attn_scale(hd)
        assert got == float(np.float32(exact)), (hd, got, exact)


def test_workload_sizes_match_oracle(orc):
    """The generator sizes its tensors with its own shape helpers; they must
    agree with the row counts the oracle derives, on all five workloads and
    on ragged variants."""
    from compressed_sparse_attention_window_gb300.workloads import WORKLOADS, TINY_PREFILL
    wls = list(WORKLOADS.values()) + [TINY_PREFILL.replace(m=m, start_pos=sp)
                                      for m in (1, 3, 17) for sp in (0, 5, 15, 16)]
    for wl in wls:
        sz = orc.step_sizes(wl.m, wl.win, wl.ratio, wl.start_pos, wl.topk)
        assert (wl.n_c, wl.G, wl.n_a, wl.K, wl.ctopk) == (
            sz["n_c"], sz["G"], sz["n_a"], sz["K"], sz["ctopk"]), wl


# ---------------------------------------------------------------------------
# Indexer (reading): dot, head-sum order, visibility, w = 0
# ---------------------------------------------------------------------------
def _q8(orc, bits):
    y, _, _ = orc.fp4_quant(bits.reshape(-1, bits.shape[-1]), 32, False)
    return orc.bf16_to_f32(y).reshape(bits.shape).astype(np.float64)


def test_indexer_single_head_is_relu_dot(orc):
    rng = np.random.default_rng(8)
    m, Hi, Di, n_c = 6, 1, 64, 9
    q = _bf16_bits_of(rng.standard_normal((m, Hi, Di)).astype(np.float32))
    k = _bf16_bits_of(rng.standard_normal((n_c, Di)).astype(np.float32))
    w = np.ones((m, Hi), np.float32)
    sc, bad = orc.indexer_scores(q, k, w, ratio=1, start_pos=3)
    assert bad == 0
    qd, kd = _q8(orc, q), _q8(orc, k)
    for t in range(m):
        vis = min(n_c, 3 + t + 1)
        dots = kd @ qd[t, 0]
        want = orc.f32_to_bf16(np.maximum(dots, 0).astype(np.float32))
        assert np.array_equal(sc[t, :vis], want[:vis])
        assert np.all(sc[t, vis:] == 0xFF80)


def _round_f32(fr: Fraction) -> float:
    """Round an exact rational to the nearest f32 (ties to even)."""
    if fr == 0:
        return 0.0
    f64 = float(fr)                       # correctly rounded to f64
    c = np.float32(f64)
    # fix double rounding: compare against both f32 neighbours exactly
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - fr),
                                     int(np.array(v, np.float32).view(np.uint32)) & 1))
    return float(best)


def test_indexer_head_sum_is_ordered_fma_chain(orc):
    rng = np.random.default_rng(9)
    m, Hi, Di, n_c = 3, 5, 32, 40
    q = _bf16_bits_of(rng.standard_normal((m, Hi, Di)).astype(np.float32))
    k = _bf16_bits_of(rng.standard_normal((n_c, Di)).astype(np.float32))
    w = rng.standard_normal((m, Hi)).astype(np.float32)
    sc, bad, acc = orc.indexer_scores(q, k, w, ratio=1, start_pos=n_c, want_acc=True)
    assert bad == 0
    qd, kd = _q8(orc, q), _q8(orc, k)
    for t in range(m):
        for s in range(n_c):
            a = 0.0
            for h in range(Hi):
                r = max(float(kd[s] @ qd[t, h]), 0.0)
                a = _round_f32(Fraction(float(w[t, h])) * Fraction(r) + Fraction(a))
            assert np.float32(a) == acc[t, s], (t, s)
            b = orc.f32_to_bf16(np.array([a], np.float32))[0]
            assert sc[t, s] == (0 if b == 0x8000 else b)


def test_indexer_zero_weights(orc):
    rng = np.random.default_rng(10)
    q = _bf16_bits_of(rng.standard_normal((4, 3, 32)).astype(np.float32))
    k = _bf16_bits_of(rng.standard_normal((12, 32)).astype(np.float32))
    sc, _ = orc.indexer_scores(q, k, np.zeros((4, 3), np.float32), ratio=2, start_pos=10)
    for t in range(4):
        vis = min(12, (10 + t + 1) // 2)
        assert np.all(sc[t, :vis] == 0) and np.all(sc[t, vis:] == 0xFF80)
    win_idx = np.full((4, 2), -1, np.int32)
    idx = orc.topk_merge(sc, win_idx, n_c=12, win=2, ratio=2, start_pos=10, topk=3, offset=100)
    for t in range(4):
        assert list(idx[t, 2:]) == [100, 101, 102]


# ---------------------------------------------------------------------------
# Pin 6: top-k by brute force over subsets
# ---------------------------------------------------------------------------
def test_topk_bruteforce_subsets(orc):
    rng = np.random.default_rng(11)
    levels = np.array([-1.5, -0.5, 0.0, 0.25, 0.5, 2.0], np.float32)
    for trial in range(300):
        n_c = int(rng.integers(1, 11))
        topk = int(rng.integers(1, 12))
        m = 3
        sp = int(rng.integers(0, n_c + 2))
        vals = levels[rng.integers(0, len(levels), (m, n_c))]
        sc = _bf16_bits_of(vals)
        win_idx = np.arange(m * 2, dtype=np.int32).reshape(m, 2)
        idx = orc.topk_merge(sc, win_idx, n_c=n_c, win=2, ratio=1, start_pos=sp, topk=topk,
                             offset=50)
        ctopk = min(topk, n_c)
        assert idx.shape == (m, 2 + ctopk)
        for t in range(m):
            assert list(idx[t, :2]) == list(win_idx[t])
            vis = min(n_c, sp + t + 1)
            k = min(ctopk, vis)
            sel = [int(v) - 50 for v in idx[t, 2:] if v >= 0]
            assert len(sel) == k and (idx[t, 2:] < 0).sum() == ctopk - k
            best = None
            for sub in itertools.combinations(range(vis), k):
                key = (sum(float(vals[t, s]) for s in sub), [-s for s in sub])
                if best is None or key > best[0]:
                    best = (key, sub)
            assert sorted(sel) == list(best[1]), (trial, t)


# ---------------------------------------------------------------------------
# Pins 7-9: sparse attention
# ---------------------------------------------------------------------------
def _dense_softmax_attn(qf, R, scale, sink=None):
    """Independent dense attention in f64: softmax over the given rows (plus a
    sink logit column when sink is given) applied to the same rows."""
    logits = scale * (qf @ R.T)
    if sink is not None:
        logits = np.concatenate([logits, np.full((logits.shape[0], 1), sink)], axis=1)
    mx = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - mx)
    p = e / e.sum(axis=1, keepdims=True)
    return p[:, : R.shape[0]] @ R


def test_sink_minus_inf_is_plain_softmax(orc):
    rng = np.random.default_rng(12)
    nh, hd, n_a, K = 3, 16, 20, 9
    q = _bf16_bits_of(rng.standard_normal((2, nh, hd)).astype(np.float32))
    ra = _bf16_bits_of(rng.standard_normal((n_a, hd)).astype(np.float32))
    idx = np.stack([rng.permutation(n_a)[:K] for _ in range(2)]).astype(np.int32)
    idx[1, 3] = -1
    sink = np.full(nh, -np.inf, np.float32)
    o, lse, bad = orc.sparse_attn(q, ra, None, idx, sink, 0.25)
    assert bad == 0
    R = orc.bf16_to_f32(ra).astype(np.float64)
    qf = orc.bf16_to_f32(q).astype(np.float64)
    for t in range(2):
        rows = R[idx[t][idx[t] >= 0]]
        want = _dense_softmax_attn(qf[t], rows, 0.25)
        assert np.allclose(o[t], want, rtol=1e-12, atol=1e-13)


def test_one_hot_row_closed_form(orc):
    nh, hd, K = 2, 8, 6
    q = np.zeros((1, nh, hd), np.float32)
    q[0, :, 2] = [1.5, -2.0]
    rows = np.zeros((K, hd), np.float32)
    rows[4, 2] = 3.0
    rows[4, 5] = -1.0
    sink = np.array([0.5, -1.0], np.float32)
    idx = np.arange(K, dtype=np.int32)[None, :]
    o, lse, _ = orc.sparse_attn(_bf16_bits_of(q), _bf16_bits_of(rows), None, idx, sink, 0.5)
    for h in range(nh):
        s = 0.5 * float(q[0, h, 2]) * 3.0
        den = math.exp(float(sink[h])) + math.exp(s) + (K - 1) * 1.0
        want = math.exp(s) / den * rows[4].astype(np.float64)
        assert np.allclose(o[0, h], want, rtol=1e-13, atol=1e-15)
        assert math.isclose(lse[0, h], math.log(den), rel_tol=1e-13)


def _run_pipeline(orc, wl, inp):
    """The oracle's whole forward for one workload (every token)."""
    from compressed_sparse_attention_window_gb300.workloads import bf16_bits
    b = {k: bf16_bits(inp[k]) for k in ("kv", "ring", "latent", "cache", "q_idx", "k_idx", "q")}
    return orc.forward(b["kv"], b["ring"], b["latent"], b["cache"], b["q_idx"], b["k_idx"],
                       inp["w"].numpy(), b["q"], inp["sink"].numpy(), win=wl.win, ratio=wl.ratio,
                       start_pos=wl.start_pos, topk=wl.topk, rd=wl.rd)


@pytest.mark.parametrize("variant", ["prefill", "decode", "chunked"])
def test_topk_covering_all_rows_is_dense_causal(orc, variant):
    """topk >= candidate count: the sparse forward equals dense causal
    attention over the window rows and the visible compressed rows, written as
    one masked dense matrix with a sink column."""
    from compressed_sparse_attention_window_gb300.workloads import TINY_PREFILL, make_inputs
    base = TINY_PREFILL.replace(topk=64)
    wl = {"prefill": base,
          "decode": base.replace(m=1, start_pos=43),
          "chunked": base.replace(m=24, start_pos=37)}[variant]
    inp = make_inputs(wl, seed=21)
    r = _run_pipeline(orc, wl, inp)
    from compressed_sparse_attention_window_gb300.workloads import bf16_bits
    # positions -> rows, built independently: the window rows by position
    pos_rows = {}
    ring = bf16_bits(inp["ring"])
    for q in range(max(0, wl.start_pos - wl.win), wl.start_pos):
        pos_rows[q] = ring[q % wl.win]
    kv = bf16_bits(inp["kv"])
    for t in range(wl.m):
        pos_rows[wl.start_pos + t] = kv[t]
    # compressed rows complete at or before each position: counted here by
    # walking the positions, not with the oracle's arithmetic
    n_c, _ = _groups_by_enumeration(wl.m, wl.ratio, wl.start_pos)
    comp = r["cache"][:n_c]
    qf = orc.bf16_to_f32(bf16_bits(inp["q"])).astype(np.float64)
    sink = inp["sink"].numpy().astype(np.float64)
    for t in range(wl.m):
        p = wl.start_pos + t
        wpos = [q for q in range(max(0, p - wl.win + 1), p + 1)]
        vis, _ = _groups_by_enumeration(1, wl.ratio, p)
        R = np.concatenate([np.stack([pos_rows[q] for q in wpos]), comp[:vis]])
        Rf = orc.bf16_to_f32(R).astype(np.float64)
        for h in range(wl.nh):
            want = _dense_softmax_attn(qf[t, h][None, :], Rf, wl.scale, sink[h])[0]
            assert np.allclose(r["o"][t, h], want, rtol=1e-11, atol=1e-12), (variant, t, h)
