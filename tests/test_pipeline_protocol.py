"""The forward kernel's barrier protocol, checked on a CPU model (no GPU).

tests/pipeline_model.py restates the order of every wait and arrival of the
kernel's roles; here random interleavings of it must finish without a deadlock
and without any parity wait that could alias. A variant with a single P-ready
barrier per tile (an earlier protocol that let the softmax run two blocks
ahead of the PV issuer) must be caught, which shows the check has teeth.
"""
import pytest

from pipeline_model import ROWS, simulate


def _items(N, all_blocks):
    nqb = (N + ROWS - 1) // ROWS
    if not all_blocks:
        return [(nqb - 1) * ROWS]
    return [qb * ROWS for qb in range(nqb - 1, -1, -1)]  # longest first, as the kernel schedules


@pytest.mark.parametrize("N,causal", [(1000, True), (8192, True), (384, True), (200, True), (129, False),
                                      (1000, False), (64, False), (1, True)])
@pytest.mark.parametrize("ring", [2, 5, 6])
def test_protocol_completes_without_aliasing(N, causal, ring):
    for all_blocks in (False, True):
        for seed in range(6 if N <= 1000 else 2):
            assert simulate(N, causal, _items(N, all_blocks), ring, seed)


def test_single_p_barrier_is_caught():
    caught = 0
    for seed in range(10):
        try:
            simulate(1000, True, _items(1000, False), 5, seed, per_buffer_p=False)
        except AssertionError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("n_it", [1, 2, 3, 7, 32])
@pytest.mark.parametrize("stages", [2, 3])
def test_backward_protocol_completes_without_aliasing(n_it, stages):
    from pipeline_model import simulate_bwd

    for seed in range(20):
        assert simulate_bwd(n_it, stages, seed)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("ring", [2, 5])
def test_packed_batch_items_with_no_rows(causal, ring):
    """Packed batches have items whose sequence is shorter than the item's
    first row (nothing to do); the producer must not fill a K slot for them."""
    lengths = [0, 1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 0, 300]
    n_items = (max(lengths) + ROWS - 1) // ROWS
    items = [(qb * ROWS, L) for qb in range(n_items - 1, -1, -1) for L in lengths]
    for seed in range(8):
        assert simulate(max(lengths), causal, items, ring, seed)


def test_loading_k_for_an_empty_item_is_caught():
    lengths = [0, 1, 300, 0, 1000]
    items = [(qb * ROWS, L) for qb in range(3, -1, -1) for L in lengths]
    with pytest.raises(AssertionError):
        simulate(1000, True, items, 2, 0, skip_empty_items=False)


@pytest.mark.parametrize("n_it", [1, 2, 3, 5, 32])
def test_backward_half_block_protocol(n_it):
    from pipeline_model import simulate_bwd_halves

    for seed in range(20):
        for stages in (2, 3):
            assert simulate_bwd_halves(n_it, stages, seed)


def _packed_items(lengths):
    """The compact packed-batch list (longest first, no empty items)."""
    top = (max(lengths) + ROWS - 1) // ROWS
    return [(qb * ROWS, L) for qb in range(top - 1, -1, -1) for L in lengths if L > qb * ROWS]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("ring", [2, 5])
@pytest.mark.parametrize("item_ring", [1, 2, 4])
def test_packed_batch_item_ring(causal, ring, item_ring):
    """Items handed from the scheduler warp to the 13 consumer warps through the
    ring: no deadlock, no aliased parity wait, for short and empty lists."""
    for lengths in ([1000, 1, 300, 64, 257], [5], [128, 129]):
        for seed in range(6):
            assert simulate(max(lengths), causal, _packed_items(lengths), ring, seed, item_ring=item_ring)
    assert simulate(16, causal, [], ring, 0, item_ring=item_ring)  # end marker only


def test_item_ring_without_empty_wait_is_caught():
    caught = 0
    for seed in range(10):
        try:
            simulate(2000, True, _packed_items([2000, 700, 300, 1500]), 5, seed, item_ring=2,
                     ring_waits_empty=False)
        except AssertionError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("ring", [2, 5])
def test_single_tile_units(causal, ring):
    """The dense schedule may cut its last items into single query tiles (tile 1 of
    the unit has no rows while tile 0 sees every key block): two-tile items
    followed by such units complete without aliasing."""
    N = 1000
    pairs = [qb * ROWS for qb in range(3, -1, -1)]
    units = [(q0, N, min(N, q0 + 128)) for qb in range(3, -1, -1) for q0 in (qb * ROWS, qb * ROWS + 128)]
    for seed in range(8):
        assert simulate(N, causal, pairs[:2] + units[4:], ring, seed)
        assert simulate(N, causal, units, ring, seed)


# ---------------------------------------------------------------- the 128-key-block kernel
def _items128(N, all_blocks):
    nqb = (N + ROWS - 1) // ROWS
    return [qb * ROWS for qb in range(nqb - 1, -1, -1)] if all_blocks else [(nqb - 1) * ROWS]


@pytest.mark.parametrize("N,causal", [(1000, True), (4096, True), (384, True), (200, True), (129, False),
                                      (1000, False), (64, False), (1, True), (256, True), (257, False)])
@pytest.mark.parametrize("rk,rv", [(3, 2), (6, 6), (2, 2)])
def test_bk128_protocol_completes_without_hazards(N, causal, rk, rv):
    from pipeline_model import simulate_bk128

    for all_blocks in (False, True):
        for seed in range(4 if N <= 1000 else 2):
            assert simulate_bk128(N, causal, _items128(N, all_blocks), rk, rv, seed)
            # P V commits that lag several products behind
            assert simulate_bk128(N, causal, _items128(N, all_blocks), rk, rv, seed, rescale_prob=0.3,
                                  late_weight=0.05)


def test_bk128_single_tile_units_and_packed_items():
    """Single-tile units of the dense schedule and packed-batch items (some with no rows),
    taken from the item ring as the packed kernel does."""
    from pipeline_model import simulate_bk128

    lengths = [0, 1, 127, 128, 129, 255, 256, 257, 700, 0, 300]
    n_items = (max(lengths) + ROWS - 1) // ROWS
    packed = [(qb * ROWS, L) for qb in range(n_items - 1, -1, -1) for L in lengths]
    single = [(512, 1000, 640), (512, 1000, 1000), (768, 1000, 896), (0, 1000, 128)]
    for seed in range(4):
        assert simulate_bk128(max(lengths), True, packed, 3, 2, seed, item_ring=4)
        assert simulate_bk128(max(lengths), False, packed, 6, 6, seed, item_ring=4)
        assert simulate_bk128(1000, True, single, 3, 2, seed)


@pytest.mark.parametrize("mutation", [{"s_waits_free": False}, {"p_waits_pv": False}, {"s_issued_barriers": 1}])
def test_bk128_mutations_are_caught(mutation):
    """An S issuer that does not wait for the S buffer to be copied out, a softmax that
    stores P (or rescales O) without waiting for the previous P V product, and one
    s_issued barrier per tile instead of two (parity aliasing): each caught."""
    from pipeline_model import simulate_bk128

    caught = 0
    for seed in range(30):
        try:
            simulate_bk128(2048, False, _items128(2048, True), 3, 2, seed, rescale_prob=0.3, late_weight=0.2,
                           **mutation)
        except AssertionError:
            caught += 1
    assert caught > 0


@pytest.mark.parametrize("n_it", [1, 2, 3, 5, 9])
def test_backward_two_issuer_protocol(n_it):
    """The d = 64 backward with the S/dP products on one issuing warp and the dV/dK/dQ products on
    another: every interleaving of the two product queues keeps each buffer's contents right."""
    from pipeline_model import simulate_bwd_split

    for stages in (2, 3):
        for seed in range(150):
            assert simulate_bwd_split(n_it, stages, seed)


@pytest.mark.parametrize("mutation", [{"acc_waits": False}, {"qd_empty_count": 1}, {"acc_waits_dq_free": False}])
def test_backward_two_issuer_mutations_are_caught(mutation):
    from pipeline_model import Deadlock, simulate_bwd_split

    with pytest.raises((AssertionError, Deadlock)):
        for seed in range(400):
            simulate_bwd_split(6, 3, seed, **mutation)


@pytest.mark.parametrize("n_it", [1, 2, 3, 6])
def test_backward_d128_two_issuer_protocol(n_it):
    """The d = 128 backward with S^T, dV, dQ's first half on one issuing warp and dP^T, dK, dQ's second
    half on another: the aliased tensor-memory columns always hold the block their reader expects, and a
    stage's dO half, which holds dQ tiles until the gradient warps release it, is never refilled early."""
    from pipeline_model import simulate_bwd128_split

    for stages in (2, 3):
        for seed in range(150):
            assert simulate_bwd128_split(n_it, stages, seed)


@pytest.mark.parametrize("mutation", [{"sp_count": 1}, {"dq_count": 1}, {"q_empty_count": 1},
                                      {"waits_dq_free": False}, {"do_empty_count": 7},
                                      {"release_after_read": False}])
def test_backward_d128_two_issuer_mutations_are_caught(mutation):
    from pipeline_model import Deadlock, simulate_bwd128_split

    with pytest.raises((AssertionError, Deadlock)):
        for seed in range(400):
            simulate_bwd128_split(5, 2, seed, **mutation)
