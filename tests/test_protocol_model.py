"""The attention kernels' hand-off protocols under random schedules (tests/protocol_model.py):
the protocols the kernels use have no race; the two dQ variants that raced on the GPU, and
planted mistakes in the dK/dV and forward orders, are caught."""
from protocol_model import find_violation


def test_kernel_protocol_has_no_race():
    """Warp 1 issues S and dP, warp 2 dQ; stored dS tiles counted by parity (the kernel)."""
    assert find_violation("split", ds_by_parity=True, runs=1500, tiles=12) is None
    # runs of items: each item's first dQ product overwrites the accumulator that the
    # warps' epilogue of the item before reads
    assert find_violation("split", ds_by_parity=True, runs=600, items=True) is None


def test_dq_epilogue_after_next_dS_is_caught():
    """A planted mistake: a warp reading an item's dQ only after storing the next item's first
    dS lets that item's first dQ product overwrite the accumulator before the read."""
    v = find_violation("split", ds_by_parity=True, runs=200, items=True, late_epilogue=True)
    assert v is not None and "epilogue of item" in v, v


def test_summed_ds_count_races():
    """One count of stored dS tiles summed over the warps (the kernel before the fix): the dQ
    product can read a lagging warp's lanes before its dS is written."""
    v = find_violation("split", ds_by_parity=False, runs=400)
    assert v is not None and "dQ(" in v, v


def test_rearranged_split_races_with_summed_counts():
    """Warp 1 issuing S and dQ, warp 2 dP, with summed counts (the rearrangement that gave
    non-finite dQ on the GPU)."""
    assert find_violation("rearranged", ds_by_parity=False, runs=400) is not None
    # counting dS by parity alone leaves the S-read count summed: dP(g) can overwrite a
    # lagging warp's S(g - 1)
    v = find_violation("rearranged", ds_by_parity=True, read_by_parity=False, runs=400)
    assert v is not None and " S(" in v, v


def test_rearranged_split_with_both_counts_by_parity():
    """With both counts kept by parity the rearrangement passes the model too."""
    assert find_violation("rearranged", ds_by_parity=True, read_by_parity=True, runs=1500, tiles=12) is None
    assert find_violation("rearranged", ds_by_parity=True, read_by_parity=True, runs=600, items=True) is None


def test_dkdv_protocol_has_no_race():
    """The dK/dV kernel: one issuer, products dV(t), S^T(t + 1), dK(t), dP^T(t + 1)."""
    from protocol_model import find_violation_dkdv
    assert find_violation_dkdv(runs=1500, tiles=12) is None
    assert find_violation_dkdv(runs=600, items=True) is None
    # a planted mistake: S^T(t + 1) before dV(t) overwrites P^T(t) before it is read
    v = find_violation_dkdv(swap_order=True, runs=100)
    assert v is not None and "dV(" in v, v


def test_forward_protocol_has_no_race():
    """The forward kernel over runs of items, in each of its modes and both stage-ring depths:
    half 0 signalled by stage releases outside the fused contiguous / zigzag ring, its
    O-ready commit after the release of the item's last stage."""
    from protocol_model import find_violation_fwd
    for mode in ("single", "fused", "striped"):
        for nstage in (2, 4):
            assert find_violation_fwd(mode, runs=300, nstage=nstage) is None, (mode, nstage)


def test_forward_o_ready_before_release_races():
    """With half 0's O-ready commit before the release of the item's last stage (the kernel's
    earlier order), half 0 can finish its epilogue and take the next item's first stage-release
    wait on that stage's buffer a phase early (two stage buffers), and read a stale S."""
    from protocol_model import find_violation_fwd
    for mode in ("single", "striped"):
        v = find_violation_fwd(mode, o_after_release=False, runs=300, nstage=2)
        assert v is not None and "half 0" in v and " S(" in v, v


def test_forward_planted_early_qk_is_caught():
    """A planted mistake: the next Q K^T before the P V that reads P."""
    from protocol_model import find_violation_fwd
    v = find_violation_fwd("single", pv_late=True, runs=100)
    assert v is not None and "PV_" in v, v


def test_dkdv_epilogue_after_next_p_is_caught():
    """A planted mistake: a warp reading an item's dK/dV only after writing the next item's
    first P^T lets that item's first dV product overwrite the accumulator before the read."""
    from protocol_model import find_violation_dkdv
    v = find_violation_dkdv(runs=200, items=True, late_epilogue=True)
    assert v is not None and "epilogue of item" in v, v
