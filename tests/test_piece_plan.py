"""The data gradients' piece plans (coda_dgrad_piece_plan), checked on the CPU.

Waits in a pieced launch end only if the plan and the deal keep three rules:
every piece of every cut tile is dealt exactly once; an owner (the last piece
of a tile) is the last item of its CTA pair and no pair holds two; and the
levelling pieces of the pairs that hold a whole tile fewer are never owners.
The row-statistic launch must also cut whole row blocks only.  This test asks
the library for the plans of many shapes and pair counts, deals the pieces the
way the kernel's PieceWork does (a copy of its arithmetic), and checks those
rules, the partial-slot bounds and the piece sizes; and it pins the plans of the
Llama shapes on 76 pairs."""

import random

import pytest


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    from gemm_epilogue_fusion_gemm0_gb300 import binding as B

    return B


def deal(plan, num_tiles, npairs, nk, pair):
    """The items of one CTA pair after its whole tiles: (tile, piece, first k-block,
    end k-block, is owner), as the kernel's PieceWork hands them out."""
    dp, P, lvl_first, lvl = plan
    R = num_tiles - dp
    lvl_units = (npairs - lvl_first) * lvl
    rr_units = R * P - lvl_units
    items, i, j = [], 0, 0
    while True:
        if pair >= lvl_first and i < lvl:
            u = (pair - lvl_first) * lvl + i
            i += 1
        else:
            v = pair + j * npairs
            if v >= rr_units:
                break
            j += 1
            u = lvl_units + v
        q = u // R
        items.append((dp + u - q * R, q, q * nk // P, (q + 1) * nk // P, q == P - 1))
    return items


def check_plan(plan, M, d, N1, npairs, tile_local):
    mt, nt, nk = -(-M // 256), -(-d // 256), -(-N1 // 64)
    num_tiles = mt * nt
    slots = min(3 * num_tiles, 192)
    dp, P, lvl_first, lvl = plan
    R = num_tiles - dp
    assert 0 <= dp < num_tiles and 1 <= R <= npairs and P >= 2
    assert nk // P >= 16 and R * (P - 1) <= slots
    if not tile_local:
        assert dp % nt == 0, "the row statistic needs whole row blocks cut"
    assert 0 <= lvl_first <= npairs and lvl >= 0
    assert (npairs - lvl_first) * lvl <= (P - 1) * R, "levelling pieces would include owners"
    seen = set()
    for p in range(npairs):
        items = deal(plan, num_tiles, npairs, nk, p)
        owners = [k for k, it in enumerate(items) if it[4]]
        assert len(owners) <= 1 and (not owners or owners[0] == len(items) - 1), (p, items)
        if p >= lvl_first:
            assert not any(it[4] for it in items[:lvl])
        for tile, q, kb0, kb1, owner in items:
            assert (tile, q) not in seen
            seen.add((tile, q))
            assert dp <= tile < num_tiles and 0 <= kb0 < kb1 <= nk
            if not owner:
                assert ((tile - dp) * (P - 1) + q) * 2 + 1 < 2 * slots
    assert seen == {(t, q) for t in range(dp, num_tiles) for q in range(P)}


def test_random_shapes_keep_the_deal_rules(lib):
    rng = random.Random(1)
    planned = {False: 0, True: 0}
    for _ in range(1500):
        M = rng.randint(1, 40000)
        d = 8 * rng.randint(1, 1000)
        N1 = 8 * rng.randint(1, 12000)
        npairs = rng.choice([76, 74, 66, 60, 38, 16])
        for tile_local in (False, True):
            plan = lib.coda_dgrad_piece_plan(M, d, N1, npairs, tile_local)
            if plan is not None:
                planned[tile_local] += 1
                check_plan(plan, M, d, N1, npairs, tile_local)
    assert planned[False] > 50 and planned[True] > 50, planned


def test_llama_plans_on_76_pairs(lib):
    # row statistic: llama7b and llama70b keep whole tiles (74 % full last wave); llama1b
    # cuts its last 4 row blocks (8 tiles each) into 2 pieces, the 4 pairs with a whole tile
    # fewer taking 2 pieces each first
    assert lib.coda_dgrad_piece_plan(8192, 4096, 28672, 76) is None
    assert lib.coda_dgrad_piece_plan(4096, 8192, 57344, 76) is None
    assert lib.coda_dgrad_piece_plan(8192, 2048, 16384, 76) == (224, 2, 72, 2)
    # tile-local (SwiGLU backward): llama7b cuts its last 56 tiles into 4 pieces after 6
    # whole waves, with no levelling
    assert lib.coda_dgrad_piece_plan(8192, 4096, 28672, 76, True) == (456, 4, 76, 0)
    for shape in [(8192, 4096, 28672), (8192, 2048, 16384), (4096, 8192, 57344)]:
        plan = lib.coda_dgrad_piece_plan(*shape, 76, True)
        assert plan is not None
        check_plan(plan, *shape, 76, True)
    check_plan(lib.coda_dgrad_piece_plan(8192, 2048, 16384, 76), 8192, 2048, 16384, 76, False)


def test_invalid_arguments_are_refused(lib):
    with pytest.raises(ValueError):
        lib.coda_dgrad_piece_plan(128, 12, 512, 76)  # d not a multiple of 8
    with pytest.raises(ValueError):
        lib.coda_dgrad_piece_plan(128, 256, 512, 0)
    assert lib.coda_dgrad_piece_plan(128, 256, 512, 76) is None  # one tile: nothing to cut
