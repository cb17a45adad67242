"""The forward kernel's unit schedule, read through the library's host-only
diagnostic (the same functions the kernel runs to pick its units): every order
deals every unit exactly once, the predicted time of the busiest CTA is what a
plain recount of the dealt units gives, and the automatic choice is never worse
than the fixed orders.  No GPU: the schedule is host arithmetic."""
import numpy as np
import pytest

import exact_tiled_attention_16_gb300 as pkg

HEADS, ZIGZAG, GROUPS = 0, 1, 2


@pytest.fixture(autouse=True)
def _restore_auto_order():
    yield
    pkg.diag_force_fwd_order(-1)


def unit_blocks(u, P, N):
    """K/V blocks tile 0 and tile 1 of causal unit u visit (Nq = Nk = N, no
    offsets): unit u = head * P + r, r = 0 the heaviest pair (the last rows)."""
    nb = (N + 127) // 128
    pair = P - 1 - u % P
    out = []
    for t in (0, 1):
        last_row = min((2 * pair + t) * 128 + 127, N - 1)
        out.append(min(nb, last_row // 128 + 1))
    return out


def recount_makespan(seq, P, N):
    worst = 0.0
    for row in seq:
        t = sum(max(unit_blocks(int(u), P, N)) + 2.0 for u in row if u >= 0)
        worst = max(worst, t)
    return worst


SHAPES = [(1, 128), (2, 640), (7, 2304), (150, 1024), (80, 777), (152, 640), (608, 512), (32, 16384), (33, 4100)]
FORCED = [(HEADS, 0), (ZIGZAG, 0), (GROUPS, 1), (GROUPS, 3), (GROUPS, 7), (GROUPS, 0)]


@pytest.mark.parametrize("num_sms", [152, 7, 1000])
@pytest.mark.parametrize("order", FORCED, ids=["heads", "zigzag", "groups1", "groups3", "groups7", "groups_all"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"BH{b}N{n}" for b, n in SHAPES])
def test_every_order_deals_every_unit_once(shape, order, num_sms):
    BH, N = shape
    P = (N + 255) // 256
    pkg.diag_force_fwd_order(*order)
    info, seq = pkg.diag_fwd_schedule(BH, N, N, True, num_sms=num_sms)
    assert info["order"] == order[0]
    assert 1 <= info["grid"] <= num_sms and seq.shape == (info["grid"], info["rounds"])
    units = seq[seq >= 0]
    assert np.array_equal(np.sort(units), np.arange(BH * P)), "a unit is missing or dealt twice"
    # -1 only after a CTA's last unit; -2 (a skipped iteration) only in zigzag's odd middle pairs
    for row in seq:
        done = np.nonzero(row == -1)[0]
        if done.size:
            assert (row[done[0]:] == -1).all()
    if order[0] != ZIGZAG:
        assert not (seq == -2).any()
    else:
        assert (seq == -2).sum() == (BH if P % 2 else 0)
    assert info["makespan"] == round(recount_makespan(seq, P, N))


@pytest.mark.parametrize("shape", [(32, 16384), (32, 8192), (32, 4096), (64, 2048), (256, 4096), (8, 32768),
                                   (2, 128), (64, 16384), (48, 8192), (5, 3000)])
def test_automatic_order_is_no_worse_than_the_fixed_ones(shape):
    """Against head-major, zigzag, groups of one head and (when every head's K/V
    fits the L2 cap together) one group of all heads."""
    BH, N = shape
    auto, seq = pkg.diag_fwd_schedule(BH, N, N, True)
    fixed = [(HEADS, 0), (ZIGZAG, 0), (GROUPS, 1)]
    if BH * N * 512 <= 64 << 20:  # all heads' K/V under the 64 MiB cap: one group of all heads
        fixed.append((GROUPS, 0))
    for order in fixed:
        pkg.diag_force_fwd_order(*order)
        forced, _ = pkg.diag_fwd_schedule(BH, N, N, True)
        assert auto["makespan"] <= forced["makespan"], (order, auto, forced)
    pkg.diag_force_fwd_order(-1)
    if auto["order"] == GROUPS and auto["group_heads"] > 1:
        # the heads of a group keep their K and V (4 d bytes per key, d = 128) under 64 MiB
        assert auto["group_heads"] * N * 512 <= 64 << 20


def test_gate_shape_balance():
    """B1 H32 N16384 causal on 152 SMs: the combined heavy+light zigzag reaches
    ~96% (6.74 rounds of equal units); the chosen head groups reach >= 98%."""
    BH, N = 32, 16384
    P = N // 256
    info, seq = pkg.diag_fwd_schedule(BH, N, N, True)
    total = sum(max(unit_blocks(u, P, N)) + 2.0 for u in range(BH * P))
    assert info["order"] == GROUPS
    assert total / 152 / info["makespan"] >= 0.98
    pkg.diag_force_fwd_order(ZIGZAG, 0)
    z, _ = pkg.diag_fwd_schedule(BH, N, N, True)
    assert 0.95 <= total / 152 / z["makespan"] < 0.97


def test_table_rule():
    """attn_fwd's causal launches take their units from a 64-entry table in
    shared memory when every CTA's rounds fit, and may then use head groups;
    past 64 rounds, or for the other entry points, the units are computed by
    every role and only head-major or zigzag order is used."""
    info, seq = pkg.diag_fwd_schedule(32, 16384, 16384, True)
    assert info["table"] == 1 and info["rounds"] <= 64
    for BH, N in [(1024, 4096), (4096, 2048)]:  # 108 and 216 rounds of units
        info, seq = pkg.diag_fwd_schedule(BH, N, N, True)
        assert info["table"] == 0 and info["order"] in (HEADS, ZIGZAG) and info["rounds"] > 64
        assert np.array_equal(np.sort(seq[seq >= 0]), np.arange(BH * N // 256))
    info, _ = pkg.diag_fwd_schedule(32, 8192, 8192, True, table_ok=False)
    assert info["table"] == 0 and info["order"] in (HEADS, ZIGZAG)
    pkg.diag_force_fwd_order(GROUPS, 2)  # a forced order past 64 rounds runs computed
    info, _ = pkg.diag_fwd_schedule(1024, 4096, 4096, True)
    assert info["order"] == GROUPS and info["table"] == 0


def _noncausal_blocks(N, role):
    nb = (N + 127) // 128
    h = (nb + 1) // 2
    return nb if role == 0 else (h if role == 1 else nb - h)


@pytest.mark.parametrize("shape", [(32, 4096), (32, 16384), (2, 4096), (5, 3200), (64, 3000), (3, 6200)])
def test_pair_tail_schedule(shape):
    """Non-causal launches whose last round holds at most one unit per CTA pair
    split each of its units over a pair (clusters of two): the even CTA takes the
    first half of the key blocks (and merges), the odd one the second half,
    encoded as -3 - unit.  Every unit is still dealt exactly once to an even CTA
    or a whole-unit CTA, and the predicted makespan counts the halves."""
    BH, N = shape
    P = (N + 255) // 256
    U = BH * P
    info, seq = pkg.diag_fwd_schedule(BH, N, N, False)
    G = info["grid"]
    full, rem = divmod(U, G)
    assert info["pair_tail"] == 1 and G % 2 == 0
    assert 0 < rem <= G // 2
    whole = seq[:, :full]
    tail = seq[:, full] if seq.shape[1] > full else np.full(G, -1)
    recv = tail[0::2]
    send = tail[1::2]
    assert np.array_equal(np.sort(np.concatenate([whole[whole >= 0], recv[recv >= 0]])), np.arange(U))
    assert np.array_equal(recv[:rem], np.arange(full * G, U)) and (recv[rem:] == -1).all()
    assert np.array_equal(send[:rem], -3 - recv[:rem]) and (send[rem:] == -1).all()
    worst = 0.0
    for c in range(G):
        t = sum(_noncausal_blocks(N, 0) + 2.0 for u in seq[c, :full] if u >= 0)
        if seq.shape[1] > full and seq[c, full] != -1:
            t += _noncausal_blocks(N, 1 + (c & 1)) + 2.0
        worst = max(worst, t)
    assert info["makespan"] == round(worst)


def test_pair_tail_only_when_the_last_round_fits_the_pairs():
    # B1 H32 N8192: 1024 units = 6 rounds of 152 + 112 > 76 pairs: no pair tail
    assert pkg.diag_fwd_schedule(32, 8192, 8192, False)[0]["pair_tail"] == 0
    # too few key blocks for the split to pay (its fixed cost, measured): at least 24
    # at d = 128, 48 at d = 64
    assert pkg.diag_fwd_schedule(64, 2048, 2048, False)[0]["pair_tail"] == 0
    assert pkg.diag_fwd_schedule(64, 3000, 3000, False)[0]["pair_tail"] == 1
    assert pkg.diag_fwd_schedule(32, 4096, 4096, False, d=64)[0]["pair_tail"] == 0
    assert pkg.diag_fwd_schedule(32, 16384, 16384, False, d=64)[0]["pair_tail"] == 1
    # a single key block cannot be split; causal launches and other entry points keep whole units
    assert pkg.diag_fwd_schedule(200, 128, 128, False)[0]["pair_tail"] == 0
    assert pkg.diag_fwd_schedule(32, 4096, 4096, True)[0]["pair_tail"] == 0
    assert pkg.diag_fwd_schedule(32, 4096, 4096, False, table_ok=False)[0]["pair_tail"] == 0
    pkg.diag_set_pair_tail(False)
    try:
        assert pkg.diag_fwd_schedule(32, 4096, 4096, False)[0]["pair_tail"] == 0
    finally:
        pkg.diag_set_pair_tail(True)
    assert pkg.diag_fwd_schedule(32, 4096, 4096, False)[0]["pair_tail"] == 1


@pytest.mark.parametrize("shape", [(16, 8192), (2, 6200), (7, 6400), (32, 8192), (16, 16384)])
def test_fp8_pair_tail(shape):
    """attn_fwd_fp8 computes its units (no table, head-major for non-causal) and
    splits its last round the same way when it fits the pairs; its K/V rows are
    2 d bytes a key, so it wants at least 48 key blocks, like d = 64."""
    BH, N = shape
    P = (N + 255) // 256
    U = BH * P
    info, seq = pkg.diag_fwd_schedule(BH, N, N, False, fp8=True)
    assert info["table"] == 0 and info["order"] == HEADS
    G = info["grid"]
    full, rem = divmod(U, G)
    want = 0 < rem <= G // 2 and N >= 48 * 128
    assert info["pair_tail"] == int(want)
    units = seq[seq >= 0]
    assert np.array_equal(np.sort(units), np.arange(U))
    if want:
        assert np.array_equal(seq[1::2, full][:rem], -3 - np.arange(full * G, U))
    # too few key blocks, causal, or pair tail switched off: whole units
    assert pkg.diag_fwd_schedule(32, 4096, 4096, False, fp8=True)[0]["pair_tail"] == 0
    assert pkg.diag_fwd_schedule(BH, N, N, True, fp8=True)[0]["pair_tail"] == 0
    pkg.diag_set_pair_tail(False)
    try:
        assert pkg.diag_fwd_schedule(BH, N, N, False, fp8=True)[0]["pair_tail"] == 0
    finally:
        pkg.diag_set_pair_tail(True)


def test_noncausal_and_bad_arguments():
    pkg.diag_set_pair_tail(False)
    try:
        info, seq = pkg.diag_fwd_schedule(4, 1000, 1000, False)
    finally:
        pkg.diag_set_pair_tail(True)
    assert info["order"] == HEADS and info["table"] == 1
    # the non-causal table (beside the O staging buffers) holds 48 rounds
    assert pkg.diag_fwd_schedule(152 * 48, 256, 256, False)[0]["table"] == 1
    assert pkg.diag_fwd_schedule(152 * 48 + 1, 256, 256, False)[0]["table"] == 0
    assert np.array_equal(np.sort(seq[seq >= 0]), np.arange(4 * 4))
    with pytest.raises(pkg.AttnError):
        pkg.diag_fwd_schedule(0, 10, 10, True)
    # a launch kind outside 0 (other entry points), 1 (BF16), 2 (FP8)
    import ctypes
    import exact_tiled_attention_16_gb300._lib as L
    info = (ctypes.c_int * 7)()
    lib = pkg.load_library()
    for kind in (-1, 3):
        assert lib.attn_diag_fwd_schedule(4, 1000, 1000, 0, 0, 0, 512, kind, 152,
                                          ctypes.cast(info, ctypes.c_void_p), None, 0) == L.ATTN_ERR_DIMS
    assert lib.attn_diag_fwd_schedule(4, 1000, 1000, 0, 0, 0, 512, 2, 152,
                                      ctypes.cast(info, ctypes.c_void_p), None, 0) == 0
    with pytest.raises(pkg.AttnError):
        pkg.diag_force_fwd_order(5, 0)
