"""Pins of the oracle's output side of the layer (compress.rs, attention_any
after sparse_attn): inverse RoPE of o at each token's position, the grouped
wo_a projection rounded to bf16, then linear_bf16 with wo_b.

Each pin checks the oracle against something other than its own formula: a
worked example done by hand, the forward rotation it must undo, a single
group that must reproduce the grouped form with block-diagonal weights, exact
scaling by powers of two, bf16 ties whose rounding the definition fixes, and
numpy's matrix product with torch's bf16 rounding on sizes where no two
dimensions are equal.
"""
import numpy as np
import torch


def _bits(x):
    """float array -> bf16 bit patterns (torch's round to nearest even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _table(rd, n_pos, seed=0):
    """A RoPE table [n_pos, rd/2, 2] of (cos a, sin a) for arbitrary angles."""
    a = np.random.default_rng(seed).uniform(-np.pi, np.pi, (n_pos, rd // 2))
    return np.stack([np.cos(a), np.sin(a)], -1).astype(np.float32)


def test_out_proj_worked_example(orc):
    """One token, one head of 4 dims, rd = 2, at position 1 where the table
    holds a quarter turn (cos 0, sin 1).  Rotating back by a quarter turn maps
    the rotary pair (3, 5) to (5, -3), so o becomes (1, 2, 5, -3).  Rows
    (1,0,0,0) and (0,0,1,1) of wo_a give og = (1, 2), and wo_b = (1, 0.5)
    gives out = 1 + 1 = 2."""
    fc = np.zeros((2, 1, 2), np.float32)
    fc[0, 0] = (1, 0)
    fc[1, 0] = (0, 1)
    o = _bits(np.array([[[1, 2, 3, 5]]], np.float32))
    wo_a = _bits(np.array([[1, 0, 0, 0], [0, 0, 1, 1]], np.float32))
    wo_b = _bits(np.array([[1, 0.5]], np.float32))
    og, out = orc.attn_out_proj(o, fc, wo_a, wo_b, rd=2, groups=1, start_pos=1)
    assert np.array_equal(_f(og), [[1, 2]])
    assert np.array_equal(out, [[2.0]])


def test_out_proj_undoes_the_forward_rotation(orc):
    """o rotated forward at position p (the oracle's own forward rotation,
    pinned by the RoPE tests) projects like the unrotated values with no
    rotary dims at all: the inverse uses the same table column with the
    opposite angle.  Values are small integers so that both rotations stay
    within one f32 rounding of exact."""
    rng = np.random.default_rng(1)
    m, nh, hd, rd, groups, o_rank, dim = 3, 4, 16, 8, 2, 5, 7
    start_pos = 5
    fc = _table(rd, start_pos + m)
    x = rng.integers(-4, 5, (m, nh, hd)).astype(np.float32)
    rows = x.reshape(m * nh, hd)
    pos = np.repeat(np.arange(start_pos, start_pos + m), nh)
    rotated = orc.apply_rotary(rows, rd, pos, fc).reshape(m, nh, hd)
    # bf16 inputs: keep only rotations that bf16 holds closely enough, then
    # compare with the plain projection of x
    wa = _bits(rng.integers(-2, 3, (groups * o_rank, nh * hd // groups)))
    wb = _bits(rng.integers(-2, 3, (dim, groups * o_rank)))
    og_plain, out_plain = orc.attn_out_proj(_bits(x), fc, wa, wb, rd=0, groups=groups,
                                            start_pos=start_pos)
    og_rot, out_rot = orc.attn_out_proj(_bits(rotated), fc, wa, wb, rd=rd, groups=groups,
                                        start_pos=start_pos)
    # the bf16 rounding of the rotated values moves each product by < 2^-8
    # relative, so og agrees to within a few bf16 steps of its own size
    assert np.allclose(_f(og_rot), _f(og_plain), rtol=3e-2, atol=0.3)
    # a wrong direction (rotating further instead of back) misses by far
    og_wrong, _ = orc.attn_out_proj(_bits(orc.apply_rotary(rotated.reshape(m * nh, hd), rd, pos,
                                                              fc).reshape(m, nh, hd)),
                                    fc, wa, wb, rd=0, groups=groups, start_pos=start_pos)
    assert not np.allclose(_f(og_wrong), _f(og_plain), rtol=3e-2, atol=0.3)


def test_out_proj_groups_are_block_diagonal(orc):
    """The grouped projection equals a single group whose wo_a is the
    block-diagonal matrix of the per-group weights: group g reads o values
    g*gw .. (g+1)*gw - 1 and writes og values g*o_rank .. (g+1)*o_rank - 1."""
    rng = np.random.default_rng(2)
    m, nh, hd, rd, groups, o_rank, dim = 2, 4, 8, 4, 4, 3, 5
    gw = nh * hd // groups
    fc = _table(rd, m)
    o = _bits(rng.standard_normal((m, nh, hd)))
    wa = rng.standard_normal((groups * o_rank, gw)).astype(np.float32)
    wb = _bits(rng.standard_normal((dim, groups * o_rank)))
    full = np.zeros((groups * o_rank, nh * hd), np.float32)
    for g in range(groups):
        full[g * o_rank:(g + 1) * o_rank, g * gw:(g + 1) * gw] = wa[g * o_rank:(g + 1) * o_rank]
    og_g, out_g = orc.attn_out_proj(o, fc, _bits(wa), wb, rd=rd, groups=groups, start_pos=0)
    og_1, out_1 = orc.attn_out_proj(o, fc, _bits(full), wb, rd=rd, groups=1, start_pos=0)
    assert np.array_equal(og_g, og_1)
    assert np.array_equal(out_g, out_1)
    # and a change inside group 1 reaches og of group 1 only
    o2 = o.copy()
    o2[0, 1, 0] ^= 0x0040
    og_c, _ = orc.attn_out_proj(o2, fc, _bits(wa), wb, rd=rd, groups=groups, start_pos=0)
    changed = np.nonzero(og_c[0] != og_g[0])[0]
    assert changed.size and np.all((changed >= o_rank) & (changed < 2 * o_rank))
    assert np.array_equal(og_c[1], og_g[1])


def test_out_proj_scales_exactly(orc):
    """out is linear in wo_b and og in wo_a: scaling either by 2^k scales the
    result by exactly 2^k (bf16 and f64 hold the scaled values exactly)."""
    rng = np.random.default_rng(3)
    m, nh, hd, rd, groups, o_rank, dim = 2, 2, 8, 4, 2, 4, 3
    fc = _table(rd, 4)
    o = _bits(rng.standard_normal((m, nh, hd)))
    wa = rng.standard_normal((groups * o_rank, nh * hd // groups)).astype(np.float32)
    wb = rng.standard_normal((dim, groups * o_rank)).astype(np.float32)
    og, out = orc.attn_out_proj(o, fc, _bits(wa), _bits(wb), rd=rd, groups=groups, start_pos=2)
    og4, out8 = orc.attn_out_proj(o, fc, _bits(4 * wa), _bits(2 * wb), rd=rd, groups=groups,
                                  start_pos=2)
    assert np.array_equal(_f(og4), 4 * _f(og))
    assert np.array_equal(out8, 8 * out)


def test_out_proj_og_rounds_ties_to_even(orc):
    """og is rounded to bf16 to nearest, ties to even: with o = (1, 2^-8, 3*2^-8,
    0) and rows picking (1 + 2^-8) and (1 + 3*2^-8), both exact sums lie halfway
    between bf16 neighbours (step 2^-7 at 1) and go to the even one: 1 and
    1 + 2^-6."""
    fc = np.tile(np.array([1, 0], np.float32), (1, 1, 1))
    o = _bits(np.array([[[1, 2 ** -8, 3 * 2 ** -8, 0]]], np.float32))
    wa = _bits(np.array([[1, 1, 0, 0], [1, 0, 1, 0]], np.float32))
    wb = _bits(np.array([[1, 0]], np.float32))
    og, out = orc.attn_out_proj(o, fc, wa, wb, rd=0, groups=1, start_pos=0)
    assert np.array_equal(_f(og), [[1.0, 1 + 2 ** -6]])
    assert np.array_equal(out, [[1.0]])


def test_out_proj_products_against_library_matmul(orc):
    """Both products against numpy's matrix product (f64) on the oracle's own
    rotated o (the rotation is pinned above), with torch's bf16 rounding for
    og: sizes chosen so that no dimension equals another (a transposed wo_a or
    wo_b, or a wrong group stride, cannot line up)."""
    rng = np.random.default_rng(5)
    m, nh, hd, rd, groups, o_rank, dim = 3, 6, 16, 8, 3, 5, 7
    start_pos = 2
    gw = nh * hd // groups
    fc = _table(rd, start_pos + m)
    o = _bits(rng.standard_normal((m, nh, hd)))
    wa = _bits(rng.standard_normal((groups * o_rank, gw)))
    wb = _bits(rng.standard_normal((dim, groups * o_rank)))
    og, out = orc.attn_out_proj(o, fc, wa, wb, rd=rd, groups=groups, start_pos=start_pos)
    pos = np.repeat(np.arange(start_pos, start_pos + m), nh)
    x = orc.apply_rotary(_f(o).astype(np.float32).reshape(m * nh, hd), rd, pos, fc, inverse=True)
    x = x.astype(np.float64).reshape(m, groups, gw)
    waf = _f(wa).reshape(groups, o_rank, gw)
    acc = np.einsum("mgi,gri->mgr", x, waf).reshape(m, groups * o_rank)
    want_og = _bits(acc.astype(np.float32))
    assert np.array_equal(og, want_og)
    assert np.allclose(out, _f(og) @ _f(wb).T, rtol=1e-12, atol=1e-12)
