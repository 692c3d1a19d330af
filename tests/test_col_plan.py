"""The column split's decomposition of the activation columns and its launch plan, on the host
(no GPU).

moe_debug_col_pieces returns, for one column range, the pieces the MOE_KERNELS_COLUMNS kernel
computes on the device (the same function).  Over all CTAs of a grid the pieces must tile the
activation index space exactly once, in order, each piece inside one segment and one group of 64
columns, with column blocks that cover its columns and stay inside the expert, and a block list
that the kernel's per-CTA buffers hold.  The plan's column ranges (moe_debug_col_plan's bounds)
must cover the columns once, stay within 16 columns of the even split (a packed plan: equal it),
and never leave a CTA with more stages than the even split's costliest one.
"""
import math

import pytest

from quantized_moe_expert_dequant_gb300 import binding as Bn
from quantized_moe_expert_dequant_gb300.workloads import ALL, Shape

MAX_PIECES, MAX_BLOCKS, MAX_COLS = 16, 64, 256   # the kernel's per-CTA limits


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()


CASES = [ALL["qwen3_stack_8bit"], ALL["e512_stack"], ALL["qwen3_layer_4bit"],
         ALL["qwen15_layer_shared"],
         Shape("small", 256, 128, 8, 2, 8, 8, 8, n_shared=1, dff_shared=128, bits_shared=4),
         Shape("ragged", 384, 192, 10, 3, 4, 4, 4),
         Shape("6-bit down", 256, 128, 8, 2, 8, 8, 6, n_shared=1, dff_shared=128, bits_shared=6),
         Shape("6-bit gate/up", 256, 128, 8, 2, 6, 6, 8),
         ALL["dots_stack_mixed"],
         Shape("fewer columns than CTAs", 64, 64, 4, 2, 8, 8, 4),
         Shape("shared only", 256, 64, 1, 0, 8, 8, 8, n_shared=2, dff_shared=128, bits_shared=8)]


def check_pieces(shape, bounds):
    """Every range's pieces: contiguous, inside one segment and group, blocks covering them."""
    K, dff, nsh, dsh = shape.top_k, shape.dff, shape.n_shared, shape.dff_shared
    bsh = shape.bits_shared if nsh else shape.bits_down
    U = K * dff + nsh * dsh
    nxt = 0
    for u0, u1 in zip(bounds[:-1], bounds[1:]):
        pieces = Bn.col_pieces(K, dff, nsh, dsh, shape.bits_down, bsh, u0, u1)
        assert u0 == nxt
        assert u1 - u0 <= MAX_COLS and len(pieces) <= MAX_PIECES
        nblocks = 0
        for seg, j0, j1, a0, blk0, nb, pb, grp in pieces:
            routed = seg < K
            width, bits = (dff, shape.bits_down) if routed else (dsh, bsh)
            cb = 32 // (8 if bits == 6 else bits)   # 6-bit codes are stored as bytes
            base = seg * dff if routed else K * dff + (seg - K) * dsh
            assert 0 <= seg < K + nsh
            assert base + j0 == u0 + a0 == nxt          # contiguous, in column order
            assert 0 <= j0 < j1 <= width and j0 // 64 == (j1 - 1) // 64 == grp
            assert blk0 == j0 // cb and blk0 * cb <= j0
            assert (blk0 + nb) * cb >= j1 and (blk0 + nb - 1) * cb < j1   # blocks cover, no more
            assert (blk0 + nb) * cb <= width
            assert pb == nblocks
            nblocks += nb
            nxt = base + j1
        assert nxt == u1
        assert nblocks <= MAX_BLOCKS
    assert nxt == U


@pytest.mark.parametrize("grid", [152, 148, 7, 1])
@pytest.mark.parametrize("shape", CASES, ids=lambda s: s.name)
def test_pieces_tile_the_columns_once(built, shape, grid):
    """The even split of the columns over `grid` CTAs, cut into pieces range by range."""
    K, dff, nsh, dsh = shape.top_k, shape.dff, shape.n_shared, shape.dff_shared
    bsh = shape.bits_shared if nsh else shape.bits_down
    U = K * dff + nsh * dsh
    bounds = [U * c // grid for c in range(grid + 1)]
    if -(-U // grid) > MAX_COLS:
        c = max(range(grid), key=lambda c: bounds[c + 1] - bounds[c])
        with pytest.raises(Bn.MoeError) as e:   # beyond the kernel's per-CTA buffers
            Bn.col_pieces(K, dff, nsh, dsh, shape.bits_down, bsh, bounds[c], bounds[c + 1])
        assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
        return
    check_pieces(shape, bounds)


def cta_stages(shape, plan, u0, u1, pack):
    """A CTA's stages in a layer when every slot names a valid expert: gate/up chunks of at most R
    row pairs (4 for the CTA's first), never across an expert, then its down stages."""
    K, dff, nsh, dsh = shape.top_k, shape.dff, shape.n_shared, shape.dff_shared
    bsh = shape.bits_shared if nsh else shape.bits_down
    chunks, x = 0, u0
    while x < u1:
        routed = x < K * dff
        width = dff if routed else dsh
        rel = x if routed else x - K * dff
        R = plan["rows_a_r"] if routed else plan["rows_a_s"]
        take = min(width - rel % width, min(R, 4) if chunks == 0 else R, u1 - x)
        chunks += 1
        x += take
    pieces = Bn.col_pieces(K, dff, nsh, dsh, shape.bits_down, bsh, u0, u1)
    nbs = plan["nbs"]
    if pack:
        down = -(-(sum(p[5] for p in pieces) + len(pieces)) // (nbs + 1))
    else:
        down = sum(-(-p[5] // nbs) for p in pieces)
    return chunks, down


@pytest.mark.parametrize("grid", [152, 148])
@pytest.mark.parametrize("shape", CASES, ids=lambda s: s.name)
def test_plan_bounds_balance_the_stages(built, shape, grid):
    U = shape.top_k * shape.dff + shape.n_shared * shape.dff_shared
    plan = Bn.col_plan(shape, grid, RING)
    b = plan["bounds"]
    assert len(b) == grid + 1 and b[0] == 0 and b[-1] == U
    assert all(b[c] <= b[c + 1] for c in range(grid))
    check_pieces(shape, b)
    even = [U * c // grid for c in range(grid + 1)]
    if plan["pack"]:                           # a packed plan keeps the even split
        assert b == even
    else:                                      # boundaries within 16 columns of the even split
        assert all(abs(b[c] - even[c]) <= 16 for c in range(grid + 1))
    cost = lambda bb: max(sum(cta_stages(shape, plan, bb[c], bb[c + 1], plan["pack"]))
                          for c in range(grid))
    assert cost(b) <= cost(even)
    # prefetch when the stages past the first ring-full fit one more; pack only without it
    unpacked = max(sum(cta_stages(shape, plan, b[c], b[c + 1], False)) for c in range(grid))
    assert plan["prefetch"] == (unpacked <= 2 * plan["stages"])
    assert plan["pack"] == (plan["nbs"] <= 2 and not plan["prefetch"])


def test_plan_bounds_qwen3_8bit(built):
    """The qwen3 8-bit stack (8 slots of 768 columns, 19 CTAs a slot, 3 blocks of 4 columns a down
    stage): the even split gives 4 CTAs of every 19 five down stages (40 columns ending a few
    columns into a new group of 64); the plan gives every CTA 4, and 6 gate/up chunks."""
    shape = ALL["qwen3_stack_8bit"]
    plan = Bn.col_plan(shape, 152, RING)
    assert plan["nbs"] == 3 and not plan["pack"] and plan["prefetch"]
    b = plan["bounds"]
    even = [6144 * c // 152 for c in range(153)]
    ev = [cta_stages(shape, plan, even[c], even[c + 1], False)[1] for c in range(152)]
    assert sorted(set(ev)) == [4, 5] and ev.count(5) == 32
    st = [cta_stages(shape, plan, b[c], b[c + 1], False) for c in range(152)]
    assert all(d == 4 for _, d in st) and all(g == 6 for g, _ in st)
    assert all(38 <= b[c + 1] - b[c] <= 42 for c in range(152))


def test_bad_arguments_are_rejected(built):
    with pytest.raises(Bn.MoeError) as e:
        Bn.col_pieces(8, 768, 0, 0, 8, 8, 6100, 6145)   # range past the columns
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG
    with pytest.raises(Bn.MoeError) as e:
        Bn.col_pieces(8, 768, 0, 0, 8, 8, 40, 39)       # range backwards
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG
    with pytest.raises(Bn.MoeError) as e:
        Bn.col_pieces(8, 768, 0, 0, 5, 5, 0, 40)        # 5-bit codes: no such format
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    with pytest.raises(Bn.MoeError) as e:
        Bn.col_pieces(8, 100, 0, 0, 8, 8, 0, 40)        # width not a multiple of 64
    assert e.value.rc == Bn.MOE_ERR_INVALID_ARG


RING = 208 * 1024   # the ring the library asks for (the device's limit is above it on GB300)


@pytest.mark.parametrize("shape", CASES, ids=lambda s: s.name)
def test_plan_stages_fit_the_ring_and_the_slab_rows(built, shape):
    grid = 152
    p = Bn.col_plan(shape, grid, RING)
    bsh = shape.bits_shared if shape.n_shared else shape.bits_down
    wide = lambda b: 8 if b == 6 else b                # 6-bit down codes are stored as bytes
    assert p["cb_r"] == 32 // wide(shape.bits_down) and p["cb_s"] == 32 // wide(bsh)
    assert 2 <= p["stages"] <= 12 and p["stages"] * p["stage_bytes"] <= RING
    assert p["stage_bytes"] % 128 == 0
    assert 1 <= p["nbs"] <= 16 and (p["nbs"] + 1) * shape.din * 4 <= p["stage_bytes"]
    # a phase-A stage of each class present: its gate and up rows; R pairs, R a power of two,
    # one warp per 2048 columns of a pair, so the warps of a stage divide the 16 consumer warps
    classes = [(p["rows_a_r"], shape.bits_gate)] if shape.top_k else []
    classes += [(p["rows_a_s"], bsh)] if shape.n_shared else []
    wpr = -(-shape.din // 1024)
    for rows, bits in classes:
        assert 2 * rows * shape.din * wide(bits) // 8 <= p["stage_bytes"]
        assert rows & (rows - 1) == 0 and 16 % (rows * wpr) == 0
    # every output row quad has exactly one owner CTA, whose quads fit its ro rows
    nq, ro = shape.din // 4, p["ro"]
    assert ro % 4 == 0 and ro <= 32
    owned = [0] * nq
    for c in range(grid):
        q0, q1 = nq * c // grid, nq * (c + 1) // grid
        assert 4 * (q1 - q0) <= ro
        for q in range(q0, q1):
            owned[q] += 1
    assert owned == [1] * nq


def test_plan_refuses_what_the_kernel_does_not_take(built):
    wide = Shape("din 8192", 8192, 128, 4, 2, 8, 8, 8)
    for shape in (wide,):
        with pytest.raises(Bn.MoeError) as e:
            Bn.col_plan(shape, 152, RING)
        assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    with pytest.raises(Bn.MoeError) as e:     # a ring too small for two stages
        Bn.col_plan(ALL["qwen3_stack_8bit"], 152, 40 * 1024)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED
    with pytest.raises(Bn.MoeError) as e:     # more CTAs than the owner's sums read
        Bn.col_plan(ALL["qwen3_stack_8bit"], 161, RING)
    assert e.value.rc == Bn.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("top_k,dff,grid", [(2, 192, 5), (1, 320, 6)])
def test_plan_bounds_are_optimal_on_small_grids(built, top_k, dff, grid):
    """An exhaustive search (memoised over (CTA, boundary)) of every placement of the inner
    boundaries within 16 columns of the even split: the plan's costliest CTA has the fewest stages
    any placement gives, here one fewer than the even split's."""
    import functools
    shape = Shape("small grid", 128, dff, 4, top_k, 8, 8, 8, seed=5)
    U = top_k * dff
    plan = Bn.col_plan(shape, grid, RING)
    assert not plan["pack"]
    even = [U * c // grid for c in range(grid + 1)]
    D = min(16, U // grid // 2)

    @functools.lru_cache(maxsize=None)
    def stages(u0, u1):
        return sum(cta_stages(shape, plan, u0, u1, False))

    @functools.lru_cache(maxsize=None)
    def fewest(c, u0):     # the least max-stages of CTAs c.. when CTA c starts at u0
        if c == grid - 1:
            return stages(u0, U)
        lo, hi = max(u0, even[c + 1] - D), min(U, even[c + 1] + D)
        return min(max(stages(u0, u1), fewest(c + 1, u1)) for u1 in range(lo, hi + 1))

    cost = lambda b: max(stages(b[c], b[c + 1]) for c in range(grid))
    assert cost(plan["bounds"]) == fewest(0, 0) == cost(even) - 1
