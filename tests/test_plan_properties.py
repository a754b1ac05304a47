"""Properties of zero_plan_create over random tensor lists (host only).

For any tensor list, rank count R, micro-batch count M, stage and shard
alignment the plan must give the layout include/zero_step.h documents:
N = sum of numels, S = ceil(N / R) rounded up to the alignment (64 when 0),
padded = R * S, the tensors' offsets as running sums, owner(i) = i / S inside
[0, N) and -1 outside, the per-rank byte formulas (2 + 2 + 12 bytes per
parameter, sharded parts counted with S) and 4 * R * S bytes of staged
scratch."""
import pytest

import zero_optimizer_step_rs_gb300 as z

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def plans(draw):
    R = draw(st.integers(1, 64))
    M = draw(st.integers(1, 256 // R))
    numels = draw(st.lists(st.one_of(st.integers(0, 300), st.integers(0, 1 << 34)),
                           min_size=0, max_size=40))
    stage = draw(st.sampled_from([1, 2]))
    align = draw(st.sampled_from([0, 4, 8, 64, 128, 1024]))
    return numels, R, M, stage, align


@hypothesis.settings(max_examples=300, deadline=None)
@hypothesis.given(plans(), st.data())
def test_plan_layout_properties(args, data):
    numels, R, M, stage, align = args
    p = z.Plan(numels, R, M, stage, align)
    a = align or 64
    N = sum(numels)
    S = -(-(-(-N // R)) // a) * a
    assert (p.N, p.S, p.padded, p.R, p.M, p.stage, p.align_elems) == (N, S, R * S, R, M, stage, a)
    offs = p.tensor_offsets()
    assert offs[0] == 0 and len(offs) == len(numels) + 1
    assert all(offs[k + 1] - offs[k] == n for k, n in enumerate(numels))
    assert p.scratch_bytes_staged == 4 * R * S
    dp, z1, z2, z3 = (p.bytes_per_rank_dp, p.bytes_per_rank_z1, p.bytes_per_rank_z2,
                      p.bytes_per_rank_z3)
    assert (dp, z1, z2, z3) == (16 * N, 4 * N + 12 * S, 2 * N + 14 * S, 16 * S)
    assert p.bytes_per_rank == (z1 if stage == 1 else z2)
    if N == 0:
        assert p.owner(0) == -1
        return
    # padding is less than one alignment unit per shard (trailing shards
    # may be empty when N is small against R * alignment)
    assert N <= R * S and S - (-(-N // R)) < a
    probes = {0, N - 1, data.draw(st.integers(0, N - 1))}
    probes |= {k * S + d for k in range(1, R) for d in (-1, 0) if 0 <= k * S + d < N}
    for i in sorted(probes)[:64]:
        assert p.owner(i) == i // S, i
    assert p.owner(-1) == -1 and p.owner(N) == -1
