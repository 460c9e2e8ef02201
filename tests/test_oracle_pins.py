"""Pins for the fp64 oracle: closed forms, special cases that reduce to library
routines, invariants and exact index-handling checks.  CPU only.

Each test fixes something the pages and the mathematics determine without
re-typing the oracle's own loop:
  * dense special case  -> scipy softmax / logsumexp over a numpy matmul
  * q = 0               -> out is the mean of the selected V rows, lse = ln(k_valid)
  * one valid entry     -> out is that V row, lse = scale * <q, K>
  * equal scores        -> uniform weights (pins the rope columns' role in K)
  * paging, padding, index order, shard split + merge, merge order -> invariances
  * one-hot V rows      -> the exact multiset of rows read
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from tests._problems import D_QK, D_V, Paged, bf16_bits, bits_to_f64, rng_normal

SCALE = 1.0 / math.sqrt(192.0)


def problem(dense, seq_lens, q, topk, Q=1, bs=64, perm_seed=None, fill=0.0, spare=0):
    pg = Paged(np.asarray(dense, np.float32), seq_lens, bs, perm_seed, spare, fill)
    q_bits = bf16_bits(q)
    prob = oracle.Problem(q_bits, pg.kv, pg.block_table, pg.seq_lens,
                          np.asarray(topk, dtype=np.int32), Q, SCALE)
    return prob, pg


def bf(x):
    """Values as the oracle sees them: rounded to bf16, widened to float64."""
    return bits_to_f64(bf16_bits(x))


# --------------------------------------------------------------------------------------
# special case: every position selected == dense softmax attention (library routines)
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("S,bs,perm", [(200, 64, None), (130, 16, 3), (64, 64, 5)])
def test_dense_equals_library_softmax_attention(S, bs, perm):
    B, h = 2, 3
    dense = rng_normal((B, S, D_QK), 1)
    q = rng_normal((B, h, D_QK), 2)
    topk = np.tile(np.arange(S, dtype=np.int32), (B, 1))
    prob, _ = problem(dense, [S] * B, q, topk, bs=bs, perm_seed=perm)
    out, lse = oracle.decode(prob)
    K = bf(dense)
    Qm = bf(q)
    for b in range(B):
        s = SCALE * (Qm[b] @ K[b].T)                    # [h, S]
        ref_out = softmax(s, axis=1) @ K[b][:, :D_V]    # V = latent columns
        np.testing.assert_allclose(out[b], ref_out, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[b], logsumexp(s, axis=1), rtol=1e-13, atol=1e-12)


# --------------------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------------------
def test_zero_query_gives_mean_of_selected_rows_and_ln_k():
    B, S, h = 2, 300, 2
    dense = rng_normal((B, S, D_QK), 11)
    q = np.zeros((B, h, D_QK), np.float32)
    rng = np.random.default_rng(12)
    sel = [rng.choice(S, size=37, replace=False), rng.choice(S, size=5, replace=False)]
    topk = np.full((B, 40), -1, np.int32)
    for b in range(B):
        topk[b, : len(sel[b])] = sel[b]
    prob, _ = problem(dense, [S] * B, q, topk, perm_seed=9)
    out, lse = oracle.decode(prob)
    K = bf(dense)
    for b in range(B):
        for hh in range(h):
            np.testing.assert_allclose(out[b, hh], K[b, sel[b], :D_V].mean(axis=0), rtol=0, atol=1e-14)
            assert lse[b, hh] == pytest.approx(math.log(len(sel[b])), abs=1e-15)


def test_single_entry_gives_that_row_and_its_scaled_score():
    S, h = 128, 4
    dense = rng_normal((1, S, D_QK), 21)
    q = rng_normal((1, h, D_QK), 22)
    p = 77
    topk = np.array([[-1, p, -1, 500]], np.int32)  # 500 is outside the cache: padding
    prob, _ = problem(dense, [S], q, topk, perm_seed=1)
    out, lse = oracle.decode(prob)
    K = bf(dense)[0, p]
    Qm = bf(q)[0]
    for hh in range(h):
        np.testing.assert_array_equal(out[0, hh], K[:D_V])
        assert lse[0, hh] == pytest.approx(SCALE * float(Qm[hh] @ K), rel=1e-14, abs=1e-14)


def test_equal_rope_scores_give_uniform_weights():
    # q lives only in the rope columns and every row has the same rope part, so
    # every score is equal: out = mean of the latent rows, lse = s + ln(n).
    S, h, n = 256, 2, 50
    dense = rng_normal((1, S, D_QK), 31)
    rope = rng_normal((D_QK - D_V,), 32)
    dense[0, :, D_V:] = rope
    q = np.zeros((1, h, D_QK), np.float32)
    q[0, :, D_V:] = rng_normal((h, D_QK - D_V), 33)
    sel = np.random.default_rng(34).choice(S, size=n, replace=False)
    prob, _ = problem(dense, [S], q, sel[None, :], perm_seed=2)
    out, lse = oracle.decode(prob)
    K = bf(dense)[0]
    Qm = bf(q)[0]
    for hh in range(h):
        s = SCALE * float(Qm[hh, D_V:] @ bf(rope))
        np.testing.assert_allclose(out[0, hh], K[sel, :D_V].mean(axis=0), rtol=0, atol=1e-13)
        assert lse[0, hh] == pytest.approx(s + math.log(n), abs=1e-13)


def test_rope_columns_enter_the_score_but_not_the_output():
    # latent part zero: out must be 0 while lse depends on the rope columns only
    S, h = 64, 2
    dense = np.zeros((1, S, D_QK), np.float32)
    dense[0, :, D_V:] = rng_normal((S, D_QK - D_V), 41)
    q = rng_normal((1, h, D_QK), 42)
    sel = np.arange(0, S, 3)
    prob, _ = problem(dense, [S], q, sel[None, :])
    out, lse = oracle.decode(prob)
    assert np.all(out == 0.0)
    s = SCALE * (bf(q)[0][:, D_V:] @ bf(dense)[0, sel, D_V:].T)
    np.testing.assert_allclose(lse[0], logsumexp(s, axis=1), rtol=1e-14)


def test_duplicate_entries_count_once_per_list_entry():
    S = 64
    dense = rng_normal((1, S, D_QK), 51)
    q = np.zeros((1, 1, D_QK), np.float32)
    prob, _ = problem(dense, [S], q, np.array([[3, 3, 7, -1]], np.int32))
    out, lse = oracle.decode(prob)
    K = bf(dense)[0]
    np.testing.assert_allclose(out[0, 0], (2 * K[3, :D_V] + K[7, :D_V]) / 3, atol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(3), abs=1e-15)


def test_empty_selection_gives_zero_and_minus_inf():
    S = 64
    dense = rng_normal((1, S, D_QK), 61)
    q = rng_normal((1, 2, D_QK), 62)
    prob, _ = problem(dense, [S], q, np.array([[-1, 64, 1000, -7]], np.int32))
    out, lse = oracle.decode(prob)
    assert np.all(out == 0.0)
    assert np.all(np.isneginf(lse))


def test_mtp_query_tokens_see_their_own_causal_range():
    # Q=2: token 0 sees [0, L-1), token 1 sees [0, L)
    L = 100
    dense = rng_normal((1, L, D_QK), 71)
    q = np.zeros((2, 1, D_QK), np.float32)
    topk = np.array([[L - 1, 0, 5], [L - 1, 0, 5]], np.int32)
    prob, _ = problem(dense, [L], q, topk, Q=2)
    out, lse = oracle.decode(prob)
    K = bf(dense)[0]
    np.testing.assert_allclose(out[0, 0], K[[0, 5], :D_V].mean(axis=0), atol=1e-14)
    np.testing.assert_allclose(out[1, 0], K[[L - 1, 0, 5], :D_V].mean(axis=0), atol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(2))
    assert lse[1, 0] == pytest.approx(math.log(3))


# --------------------------------------------------------------------------------------
# exact index handling
# --------------------------------------------------------------------------------------
def test_one_hot_rows_recover_the_exact_multiset_read():
    # q = 0 and latent row of position p = one-hot at column p % 512: out * n counts
    # how often each residue was read.  Every unselected row (and every padding
    # target) is NaN, so a stray read would poison the output.
    B, S = 2, 1024
    dense = np.full((B, S, D_QK), np.nan, np.float32)
    rng = np.random.default_rng(81)
    topk = np.full((B, 300), -1, np.int32)
    expected = np.zeros((B, D_V))
    for b in range(B):
        pos = rng.choice(S, size=256, replace=False)
        pos = pos[np.unique(pos % D_V, return_index=True)[1]][:200]
        for p in pos:
            dense[b, p] = 0.0
            dense[b, p, p % D_V] = 1.0
            expected[b, p % D_V] += 1
        topk[b, : len(pos)] = pos
        topk[b, len(pos):len(pos) + 20] = rng.integers(S, 4 * S, size=20)  # out of range
    q = np.zeros((B, 3, D_QK), np.float32)
    prob, _ = problem(dense, [S] * B, q, topk, perm_seed=4, fill=np.nan, spare=3)
    out, lse = oracle.decode(prob)
    for b in range(B):
        n = expected[b].sum()
        for hh in range(3):
            assert np.all(np.isfinite(out[b, hh]))
            np.testing.assert_array_equal(np.rint(out[b, hh] * n), expected[b])
            assert lse[b, hh] == pytest.approx(math.log(n))


def test_nan_in_unselected_rows_does_not_leak():
    B, S, h = 1, 512, 4
    dense = rng_normal((B, S, D_QK), 91)
    q = rng_normal((B, h, D_QK), 92)
    sel = np.random.default_rng(93).choice(S, size=64, replace=False)
    clean, _ = problem(dense, [S], q, sel[None, :], perm_seed=6)
    poisoned_dense = np.full_like(dense, np.nan)
    poisoned_dense[0, sel] = dense[0, sel]
    dirty, _ = problem(poisoned_dense, [S], q, sel[None, :], perm_seed=6, fill=np.nan, spare=2)
    o1, l1 = oracle.decode(clean)
    o2, l2 = oracle.decode(dirty)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# --------------------------------------------------------------------------------------
# invariances
# --------------------------------------------------------------------------------------
def _random_problem(seed, B=3, S=333, h=5, k=90, Q=1, perm=None, bs=64):
    rng = np.random.default_rng(seed)
    dense = rng.standard_normal((B, S, D_QK)).astype(np.float32)
    q = rng.standard_normal((B * Q, h, D_QK)).astype(np.float32)
    topk = np.stack([rng.choice(S, size=k, replace=False) for _ in range(B * Q)]).astype(np.int32)
    return dense, q, topk


def test_index_order_does_not_matter():
    dense, q, topk = _random_problem(101)
    p1, _ = problem(dense, [333] * 3, q, topk, perm_seed=1)
    perm = np.random.default_rng(102).permutation(topk.shape[1])
    p2, _ = problem(dense, [333] * 3, q, topk[:, perm], perm_seed=1)
    o1, l1 = oracle.decode(p1)
    o2, l2 = oracle.decode(p2)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_padding_entries_do_not_matter():
    dense, q, topk = _random_problem(111)
    rng = np.random.default_rng(112)
    pad = np.concatenate([np.full((3, 10), -1), rng.integers(333, 10 ** 6, (3, 5)),
                          rng.integers(-10 ** 6, -1, (3, 5))], axis=1).astype(np.int32)
    mixed = np.concatenate([topk, pad], axis=1)
    mixed = np.stack([row[np.random.default_rng(113 + i).permutation(len(row))] for i, row in enumerate(mixed)])
    p1, _ = problem(dense, [333] * 3, q, topk)
    p2, _ = problem(dense, [333] * 3, q, mixed)
    o1, l1 = oracle.decode(p1)
    o2, l2 = oracle.decode(p2)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_physical_block_placement_does_not_matter():
    dense, q, topk = _random_problem(121, bs=16)
    outs = []
    for perm in (None, 1, 2):
        p, _ = problem(dense, [333] * 3, q, topk, bs=16, perm_seed=perm, spare=perm or 0)
        outs.append(oracle.decode(p))
    for o, l in outs[1:]:
        np.testing.assert_array_equal(o, outs[0][0])
        np.testing.assert_array_equal(l, outs[0][1])


@pytest.mark.parametrize("n_splits", [1, 2, 3, 4, 8, 13])
def test_shard_partials_merged_equal_unsplit(n_splits):
    rng = np.random.default_rng(131)
    B, S, h, Q = 3, 400, 4, 2
    dense = rng.standard_normal((B, S, D_QK)).astype(np.float32)
    seq_lens = [400, 97, 250]
    q = rng.standard_normal((B * Q, h, D_QK)).astype(np.float32)
    topk = np.full((B * Q, 120), -1, np.int32)
    for t in range(B * Q):
        L = seq_lens[t // Q]
        sel = rng.choice(L, size=min(L, 110), replace=False)
        topk[t, : len(sel)] = sel
    prob, _ = problem(dense, seq_lens, q, topk, Q=Q, perm_seed=8)
    out, lse = oracle.decode(prob)
    op, lp = oracle.decode_splits(prob, n_splits)
    mo, ml = oracle.merge(op, lp)
    np.testing.assert_allclose(mo, out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=1e-12, atol=1e-12)
    if n_splits == 1:
        np.testing.assert_array_equal(op[0], out)
        np.testing.assert_array_equal(lp[0], lse)


def test_shard_partials_closed_form_with_zero_query():
    # q = 0: shard r's partial is the mean of its rows with lse = ln(count in shard)
    S, n = 200, 3                    # shard width ceil(200/3) = 67
    dense = rng_normal((1, S, D_QK), 141)
    sel = np.array([0, 66, 67, 133, 134, 199, 150, 10], np.int32)
    prob, _ = problem(dense, [S], np.zeros((1, 2, D_QK), np.float32), sel[None, :])
    op, lp = oracle.decode_splits(prob, n)
    K = bf(dense)[0]
    shards = [[0, 66, 10], [67, 133], [134, 199, 150]]
    for r in range(n):
        np.testing.assert_allclose(op[r, 0, 0], K[shards[r], :D_V].mean(axis=0), atol=1e-14)
        assert lp[r, 0, 0] == pytest.approx(math.log(len(shards[r])))
    mo, ml = oracle.merge(op, lp)
    np.testing.assert_allclose(mo[0, 0], K[sel, :D_V].mean(axis=0), atol=1e-14)
    assert ml[0, 0] == pytest.approx(math.log(len(sel)))


def test_empty_shards_are_zero_and_minus_inf():
    S = 256
    dense = rng_normal((1, S, D_QK), 151)
    sel = np.array([[200, 201, 255]], np.int32)   # all in the last of 4 shards of 64
    prob, _ = problem(dense, [S], rng_normal((1, 1, D_QK), 152), sel)
    op, lp = oracle.decode_splits(prob, 4)
    for r in range(3):
        assert np.all(op[r] == 0) and np.all(np.isneginf(lp[r]))
    assert np.isfinite(lp[3]).all()


def test_merge_identity_order_and_empty_partials():
    rng = np.random.default_rng(161)
    op = rng.standard_normal((4, 6, D_V))
    lp = rng.standard_normal((4, 6)) * 3
    lp[1, 2] = -np.inf
    lp[:, 5] = -np.inf                                 # a row with no data at all
    one_o, one_l = oracle.merge(op[:1], lp[:1])
    np.testing.assert_array_equal(one_o[:5], op[0, :5])     # identity on rows with data
    np.testing.assert_array_equal(one_l, lp[0])
    assert np.all(one_o[5] == 0)                              # an empty partial carries no output
    mo, ml = oracle.merge(op, lp)
    perm = [2, 0, 3, 1]
    po, pl = oracle.merge(op[perm], lp[perm])
    np.testing.assert_allclose(po, mo, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(pl, ml, rtol=1e-14, atol=1e-14)
    assert np.all(mo[5] == 0) and np.isneginf(ml[5])
    # closed form: lse = logsumexp over partials, weights = softmax of the lse
    w = softmax(lp[:, :5], axis=0)
    np.testing.assert_allclose(ml[:5], logsumexp(lp[:, :5], axis=0), rtol=1e-14)
    np.testing.assert_allclose(mo[:5], np.einsum("rx,rxc->xc", w, op[:, :5]), rtol=1e-12, atol=1e-13)


def test_thread_count_does_not_change_results():
    dense, q, topk = _random_problem(171, B=4, h=8)
    prob, _ = problem(dense, [333] * 4, q, topk, perm_seed=3)
    o1, l1 = oracle.decode(prob, nthreads=1)
    o7, l7 = oracle.decode(prob, nthreads=7)
    np.testing.assert_array_equal(o1, o7)
    np.testing.assert_array_equal(l1, l7)


def test_sampled_pairs_match_full_decode():
    dense, q, topk = _random_problem(181, B=3, h=6, Q=1)
    prob, _ = problem(dense, [333] * 3, q, topk, perm_seed=5)
    out, lse = oracle.decode(prob)
    t = np.array([0, 2, 1, 2])
    hh = np.array([5, 0, 3, 3])
    so, sl = oracle.decode_sampled(prob, t, hh)
    np.testing.assert_array_equal(so, out[t, hh])
    np.testing.assert_array_equal(sl, lse[t, hh])
    op, lp = oracle.decode_splits(prob, 3)
    r = np.array([0, 2, 1, 1])
    so, sl = oracle.decode_sampled(prob, t, hh, shards=r, n_splits=3)
    np.testing.assert_array_equal(so, op[r, t, hh])
    np.testing.assert_array_equal(sl, lp[r, t, hh])


# --------------------------------------------------------------------------------------
# latent-cache write (slot_mapping scatter)
# --------------------------------------------------------------------------------------
def _cache_and_rows(seed, num_blocks=6, bs=16, T=20):
    rng = np.random.default_rng(seed)
    kv = rng.integers(0, 1 << 16, size=(num_blocks, bs, D_QK), dtype=np.uint16)
    rows = rng.integers(0, 1 << 16, size=(T, D_QK), dtype=np.uint16)
    slots = rng.permutation(num_blocks * bs)[:T].astype(np.int32)
    slots[::5] = -1                                   # padding entries
    return kv, rows, slots


def test_kv_write_places_rows_skips_padding_and_leaves_the_rest():
    kv, rows, slots = _cache_and_rows(40)
    out = oracle.kv_write(kv, slots, rows).reshape(-1, D_QK)
    flat = kv.reshape(-1, D_QK)
    written = {int(s): t for t, s in enumerate(slots) if s >= 0}
    for s in range(flat.shape[0]):
        expect = rows[written[s]] if s in written else flat[s]
        assert np.array_equal(out[s], expect)


def test_kv_write_is_order_independent_and_idempotent():
    kv, rows, slots = _cache_and_rows(41)
    once = oracle.kv_write(kv, slots, rows)
    perm = np.random.default_rng(3).permutation(len(slots))
    assert np.array_equal(oracle.kv_write(kv, slots[perm], rows[perm]), once)
    assert np.array_equal(oracle.kv_write(once, slots, rows), once)


def test_kv_write_rejects_slots_past_the_cache_and_repeated_slots():
    kv, rows, slots = _cache_and_rows(42)
    bad = slots.copy()
    bad[3] = kv.shape[0] * kv.shape[1]
    with pytest.raises(ValueError):
        oracle.kv_write(kv, bad, rows)
    rep = slots.copy()
    rep[4] = rep[1] if rep[1] >= 0 else 0
    rep[1] = rep[4]
    with pytest.raises(ValueError):
        oracle.kv_write(kv, rep, rows)


def test_decode_after_write_reads_the_new_token_row():
    # sequence 1 gets a new token at position L (its cache grows to L + 1); its slot is
    # block_table[1, L // bs] * bs + L % bs.  Attending only to it with q = 0 returns
    # exactly the new row's latent part and lse = ln 1 = 0.
    bs, L = 16, 37
    dense = rng_normal((2, 64, D_QK), 43)
    prob, pg = problem(dense, [50, L + 1], np.zeros((2, 3, D_QK), np.float32), [[0], [0]], bs=bs,
                       perm_seed=7)
    new_row = rng_normal((1, D_QK), 44)
    slot = int(pg.block_table[1, L // bs]) * bs + L % bs
    kv2 = oracle.kv_write(pg.kv, np.array([slot], np.int32), bf16_bits(new_row))
    prob2 = oracle.Problem(bf16_bits(np.zeros((2, 3, D_QK), np.float32)), kv2, pg.block_table, pg.seq_lens,
                           np.array([[0], [L]], np.int32), 1, SCALE)
    out, lse = oracle.decode(prob2)
    for hh in range(3):
        assert np.array_equal(out[1, hh], bf(new_row[0, :D_V]))
        assert lse[1, hh] == 0.0


# --------------------------------------------------------------------------------------
# W_UV up-projection
# --------------------------------------------------------------------------------------
def test_uv_proj_equals_a_plain_loop_on_a_tiny_case():
    rng = np.random.default_rng(70)
    out = rng.standard_normal((2, 3, D_V))
    w_bits = bf16_bits(rng.standard_normal((3, D_V, 128)).astype(np.float32))
    w = bits_to_f64(w_bits)
    y = oracle.uv_proj(out, w_bits)
    for t in range(2):
        for hh in range(3):
            for v in (0, 1, 77, 127):
                acc = 0.0
                for c in range(D_V):
                    acc += float(out[t, hh, c]) * float(w[hh, c, v])
                assert abs(y[t, hh, v] - acc) <= 1e-9 * (1 + abs(acc))


def test_uv_proj_identity_weights_and_linearity():
    rng = np.random.default_rng(71)
    out = rng.standard_normal((4, 2, D_V))
    eye = np.zeros((2, D_V, 128), np.float32)
    eye[:, np.arange(128), np.arange(128)] = 1.0
    assert np.array_equal(oracle.uv_proj(out, bf16_bits(eye)), out[:, :, :128])
    w_bits = bf16_bits(rng.standard_normal((2, D_V, 128)).astype(np.float32))
    a, b = rng.standard_normal((4, 2, D_V)), rng.standard_normal((4, 2, D_V))
    lhs = oracle.uv_proj(2.0 * a - b, w_bits)
    rhs = 2.0 * oracle.uv_proj(a, w_bits) - oracle.uv_proj(b, w_bits)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-9)


# --------------------------------------------------------------------------------------
# layout options: interleaved DCP shards, per-token block table
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("n_splits,g", [(2, 1), (3, 16), (4, 64), (8, 5)])
def test_interleaved_shards_merged_equal_unsplit(n_splits, g):
    rng = np.random.default_rng(90 + n_splits)
    B, S, h, Q = 3, 700, 3, 2
    dense = rng.standard_normal((B, S, D_QK)).astype(np.float32)
    seq_lens = [700, 131, 402]
    q = rng.standard_normal((B * Q, h, D_QK)).astype(np.float32)
    topk = np.full((B * Q, 210), -1, np.int32)
    for t in range(B * Q):
        L = seq_lens[t // Q]
        sel = rng.choice(L, size=min(L, 200), replace=False)
        topk[t, : len(sel)] = sel
    prob, _ = problem(dense, seq_lens, q, topk, Q=Q, perm_seed=5)
    out, lse = oracle.decode(prob)
    op, lp = oracle.decode_ex(prob, n_splits=n_splits, interleave=g)
    mo, ml = oracle.merge(op, lp)
    np.testing.assert_allclose(mo, out, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=1e-12, atol=1e-12)


def test_interleaved_shard_partials_closed_form_with_zero_query():
    # q = 0: shard r's partial is the mean of the selected V rows whose position p has
    # (p // g) % n == r, and its lse is ln(count); no such row -> (0, -inf)
    n, g, S = 3, 8, 200
    dense = rng_normal((1, S, D_QK), 91)
    topk = np.random.default_rng(92).permutation(S)[:77][None, :]
    prob, _ = problem(dense, [S], np.zeros((1, 2, D_QK), np.float32), topk, perm_seed=3)
    op, lp = oracle.decode_ex(prob, n_splits=n, interleave=g)
    V = bf(dense[0, :, :D_V])
    for r in range(n):
        sel = [p for p in topk[0] if (p // g) % n == r]
        for hh in range(2):
            if sel:
                assert np.allclose(op[r, 0, hh], V[sel].mean(axis=0), rtol=0, atol=1e-12)
                assert abs(lp[r, 0, hh] - math.log(len(sel))) < 1e-12
            else:
                assert np.all(op[r, 0, hh] == 0) and np.isneginf(lp[r, 0, hh])


def test_block_table_per_token_reads_each_tokens_own_row():
    # two query tokens of one sequence (Q = 2); token 0's row points at a copy of the
    # sequence's blocks holding different data: each token must read through its own row
    bs, S = 16, 64
    dense = rng_normal((2, S, D_QK), 93)               # "sequence" 0 and an alternative copy
    pg = Paged(dense, [S, S], bs)                       # blocks of both, one table row each
    q = rng_normal((2, 3, D_QK), 94)
    topk = np.tile(np.arange(0, S - 1, 3, dtype=np.int32), (2, 1))
    # per-sequence table: both tokens read sequence 0
    per_seq = oracle.Problem(bf16_bits(q), pg.kv, pg.block_table[:1], np.array([S], np.int32), topk, 2, SCALE)
    o_seq, l_seq = oracle.decode(per_seq)
    # per-token table: token 0 reads the alternative copy, token 1 sequence 0
    tok_bt = np.stack([pg.block_table[1], pg.block_table[0]])
    per_tok = oracle.Problem(bf16_bits(q), pg.kv, tok_bt, np.array([S], np.int32), topk, 2, SCALE)
    o_tok, l_tok = oracle.decode_ex(per_tok, bt_per_token=True)
    assert np.array_equal(o_tok[0, 1], o_seq[1]) and np.array_equal(l_tok[0, 1], l_seq[1])
    # token 0 through the alternative copy equals a per-sequence problem on that copy
    alt = oracle.Problem(bf16_bits(q), pg.kv, pg.block_table[1:], np.array([S], np.int32), topk, 2, SCALE)
    o_alt, l_alt = oracle.decode(alt)
    assert np.array_equal(o_tok[0, 0], o_alt[0]) and not np.allclose(o_tok[0, 0], o_seq[0])
    # identical rows for both tokens give exactly the per-sequence result
    same = oracle.Problem(bf16_bits(q), pg.kv, np.stack([pg.block_table[0]] * 2), np.array([S], np.int32),
                          topk, 2, SCALE)
    o_same, l_same = oracle.decode_ex(same, bt_per_token=True)
    assert np.array_equal(o_same[0], o_seq) and np.array_equal(l_same[0], l_seq)


def _problem_with_per_token_table(seed):
    # B = 2 sequences of Q = 2 tokens; each token reads its own copy of its sequence's
    # cache (4 dense copies with different data), positions drawn causally
    bs, S, Q = 16, 90, 2
    dense = rng_normal((4, S, D_QK), seed)
    pg = Paged(dense, [S] * 4, bs, perm_seed=seed + 1)
    q = rng_normal((4, 6, D_QK), seed + 2)
    rng = np.random.default_rng(seed + 3)
    topk = np.full((4, 40), -1, np.int32)
    for t in range(4):
        L = S - (Q - 1 - t % Q)
        topk[t, :37] = rng.choice(L, 37, replace=False)
    return oracle.Problem(bf16_bits(q), pg.kv, pg.block_table, np.array([S, S], np.int32), topk, Q, SCALE)


def test_sampled_layout_options_agree_with_the_whole_grid():
    """The sampled entry point with interleaved shards and a per-token table returns the
    same values as the whole-grid entry point for the same (shard, token, head)."""
    prob = _problem_with_per_token_table(seed=77)
    n, g = 3, 5
    op, lp = oracle.decode_ex(prob, n, interleave=g, bt_per_token=True)
    rng = np.random.default_rng(3)
    tt = rng.integers(0, prob.T, 20).astype(np.int32)
    hh = rng.integers(0, prob.h, 20).astype(np.int32)
    rr = rng.integers(0, n, 20).astype(np.int32)
    so, sl = oracle.decode_sampled(prob, tt, hh, shards=rr, n_splits=n, interleave=g, bt_per_token=True)
    np.testing.assert_array_equal(so, op[rr, tt, hh])
    np.testing.assert_array_equal(sl, lp[rr, tt, hh])


# ---------------------------------------------------------------------------------
# indexer top-k selection ("vllm-ascend PR #18870 解读", 4.5: sparse attention visits
# only the top-2048 positions the indexer chose)


def _numpy_topk_row(row, L, k):
    """numpy's own sort: larger score first, ties lower position first (lexsort sorts by
    the last key first), then the chosen positions in ascending order, -1 padded."""
    pos = np.arange(L)
    order = np.lexsort((pos, -row[:L].astype(np.float64)))
    sel = np.sort(order[:min(k, L)])
    return np.concatenate([sel, np.full(k - sel.size, -1)]).astype(np.int32)


def test_topk_distinct_scores_match_numpy_sort():
    rng = np.random.default_rng(101)
    T, S, k = 6, 1500, 200
    sc = rng.standard_normal((T, S)).astype(np.float32)
    sc[T // 2:] = -np.abs(sc[T // 2:])            # rows of negative scores only
    got = oracle.topk(sc, k)
    for t in range(T):
        np.testing.assert_array_equal(got[t], _numpy_topk_row(sc[t], S, k))
        # and the selected set is exactly argpartition's (distinct values: unique answer)
        assert set(got[t]) == set(np.argpartition(-sc[t], k)[:k])


def test_topk_ties_take_lower_positions_first():
    rng = np.random.default_rng(102)
    T, S, k = 5, 700, 333
    sc = rng.integers(-2, 3, (T, S)).astype(np.float32) * 0.5   # five values: heavy ties
    got = oracle.topk(sc, k)
    for t in range(T):
        np.testing.assert_array_equal(got[t], _numpy_topk_row(sc[t], S, k))
    # all equal: the first k positions
    eq = np.full((2, 50), 3.25, np.float32)
    np.testing.assert_array_equal(oracle.topk(eq, 7), np.tile(np.arange(7, dtype=np.int32), (2, 1)))


def test_topk_signed_zero_infinities_and_nan_follow_total_order():
    nan = np.float32(np.nan)
    neg_nan = np.frombuffer(np.uint32(0xFFC00000).tobytes(), np.float32)[0]
    row = np.array([[np.float32(-np.inf), nan, np.float32(np.inf), 1.0, neg_nan, -0.0, 0.0, -1.0]], np.float32)
    # totalOrder: -NaN < -inf < -1 < -0 < +0 < 1 < +inf < +NaN
    assert oracle.topk(row, 1).tolist() == [[1]]
    assert oracle.topk(row, 2).tolist() == [[1, 2]]
    assert oracle.topk(row, 3).tolist() == [[1, 2, 3]]
    assert oracle.topk(row, 4).tolist() == [[1, 2, 3, 6]]          # +0 before -0
    assert oracle.topk(row, 5).tolist() == [[1, 2, 3, 5, 6]]
    assert oracle.topk(row, 6).tolist() == [[1, 2, 3, 5, 6, 7]]
    assert oracle.topk(row, 7).tolist() == [[0, 1, 2, 3, 5, 6, 7]]  # -inf above -NaN
    assert oracle.topk(row, 9).tolist() == [[0, 1, 2, 3, 4, 5, 6, 7, -1]]
    # negatives: a larger magnitude is smaller
    neg = -np.array([[3.0, 1.0, 2.0, 0.5]], np.float32)
    assert oracle.topk(neg, 2).tolist() == [[1, 3]]


def test_topk_causal_range_and_short_rows():
    rng = np.random.default_rng(103)
    B, Q, S, k = 3, 2, 300, 64
    sc = rng.standard_normal((B * Q, S)).astype(np.float32)
    seq_lens = np.array([300, 40, 1], np.int32)
    got = oracle.topk(sc, k, seq_lens=seq_lens, Q=Q, S=S)
    for t in range(B * Q):
        L = min(S, int(seq_lens[t // Q]) - (Q - 1 - t % Q))
        np.testing.assert_array_equal(got[t], _numpy_topk_row(sc[t], max(L, 0), k))
    assert np.all(got[4] == -1)                       # L = 0: nothing selected
    np.testing.assert_array_equal(got[3][:40], np.arange(40))   # L = 40 <= k: every position
    assert np.all(got[3][40:] == -1)
    # seq_lens above S are clipped to S; the row stride may exceed S
    wide = np.concatenate([sc[:2], np.full((2, 20), 1e30, np.float32)], axis=1)
    got2 = oracle.topk(wide, k, seq_lens=np.array([5000], np.int32), Q=2, S=S)
    np.testing.assert_array_equal(got2, oracle.topk(sc[:2], k))


def test_topk_brute_force_threshold_property():
    """On tiny rows, every selected score is >= every unselected one (as floats), the
    count is min(k, L), and no position repeats."""
    rng = np.random.default_rng(104)
    for trial in range(200):
        S = int(rng.integers(1, 12))
        k = int(rng.integers(1, 14))
        row = rng.integers(-3, 4, (1, S)).astype(np.float32)
        got = oracle.topk(row, k)[0]
        sel = [p for p in got if p >= 0]
        assert len(sel) == min(k, S) and len(set(sel)) == len(sel) and sel == sorted(sel)
        rest = [p for p in range(S) if p not in sel]
        if sel and rest:
            assert min(row[0, sel]) >= max(row[0, rest])
            # among the threshold value, the chosen ones are the lowest positions
            thr = min(row[0, sel])
            tie_sel = [p for p in sel if row[0, p] == thr]
            tie_rest = [p for p in rest if row[0, p] == thr]
            if tie_rest:
                assert max(tie_sel) < min(tie_rest)
