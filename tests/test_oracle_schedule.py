"""Pins for oracle/schedule.py: the guide's printed rules (golden fixtures),
ring-table properties and the paired-block workload constancy."""
import os

import numpy as np
import pytest

from oracle import schedule

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [list(map(int, ln.split())) for ln in f if ln.strip() and not ln.startswith("#")]


def test_paired_blocks_golden():
    for p_seq, r, a, b, work in _rows("paired_blocks.txt"):
        assert schedule.paired_blocks(p_seq, r) == (a, b)
        assert a + b == work                      # r + (2P_seq - 1 - r)


def test_mesh_coordinator_golden():
    for world, ph, rank, pseq, sr, hr, ns, ps, ng, pg in _rows("mesh_coordinator.txt"):
        m = schedule.mesh_coords(rank, world, ph)
        assert (m["p_seq"], m["seq_rank"], m["head_rank"], m["next_seq_rank"],
                m["prev_seq_rank"], m["next_global_rank"], m["prev_global_rank"]) == \
            (pseq, sr, hr, ns, ps, ng, pg)


def test_zigzag_tokens_golden():
    for row in _rows("zigzag_tokens.txt"):
        S, cp, c, toks = row[0], row[1], row[2], row[3:]
        assert schedule.rank_tokens(S, cp, c).tolist() == toks


@pytest.mark.parametrize("cp,blk", [(4, 128), (8, 2048), (16, 4096), (32, 4096), (64, 8192),
                                    (3, 5)])
def test_paired_block_workload_is_constant(cp, blk):
    S = 2 * cp * blk
    works = {schedule.pair_work(S, cp, c) for c in range(cp)}
    assert works == {(2 * cp - 1) * blk * blk + blk * (blk + 1)}
    # contiguous placement is imbalanced: rank c does (2c+1) b^2/2-ish work
    cont = [schedule.pair_work(S, cp, c, schedule.CONTIGUOUS) for c in range(cp)]
    assert cont == sorted(cont) and cont[0] < cont[-1]


@pytest.mark.parametrize("inner,outer", [(4, 1), (4, 2), (8, 2), (8, 4), (8, 8), (1, 5), (3, 3)])
def test_double_ring_table_properties(inner, outer):
    cp = inner * outer
    tab = schedule.schedule_table(inner, outer)
    assert tab.shape == (cp, cp)
    assert np.all(tab[0] == np.arange(cp))                  # step 0: own K/V
    for t in range(cp):
        assert sorted(tab[t]) == list(range(cp))             # every step is a bijection
    for c in range(cp):
        assert sorted(tab[:, c]) == list(range(cp))          # each rank sees each source once
    for t in range(cp):
        o, i = divmod(t, inner)
        for c in range(cp):
            g, l = divmod(c, inner)
            if i > 0:   # one hop around the inner ring since the previous step
                assert tab[t, c] == tab[t - 1, g * inner + (l - 1) % inner]
            elif o > 0:  # the round's first chunk made one hop around the outer ring
                assert tab[t, c] == tab[t - inner, ((g - 1) % outer) * inner + l]


def test_single_ring_receives_from_previous_rank():
    # "GPU i receives (K_j, V_j) from GPU i-1": with outer = 1, step t holds rank (c - t)'s K/V
    for cp in (2, 4, 7):
        for t in range(cp):
            for c in range(cp):
                assert schedule.ring_source(c, t, cp, 1) == (c - t) % cp


def test_head_group_split_and_gqa_ceiling():
    qh, kh = schedule.head_group(3, 32, 8, 8)
    assert qh == [12, 13, 14, 15] and kh == [3]
    assert all(q // 4 in kh for q in qh)
    with pytest.raises(ValueError):
        schedule.head_group(0, 32, 8, 16)        # hp > Hkv: a kv head would be split
