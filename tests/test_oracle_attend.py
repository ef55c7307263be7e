"""Pins of the block-sparse attend oracle (oracle/attend.py), and planted
mistakes each caught by one of them.

The pins: a scalar pure-Python brute force (oracle/brute.py, walking every
position of the request) on tiny inputs; closed forms (one visible token:
o = its v row exactly; a zero query: o = the mean of the visible v rows;
nothing visible: o = 0); the causal cut inside the local page; the order of
the ids in a row does not matter; -1 ids are skipped; the fp32 error bound
covers an fp32 online-softmax evaluation in page blocks and is tight enough
that dropping one visible token is outside it.
"""
import numpy as np
import pytest

import workloads
from oracle import attend as oat
from oracle import brute


def _case(seed, H=2, G=2, nreq=2, seq=(300, 700), nb=16):
    rng = np.random.Generator(np.random.PCG64(seed))
    width = max((s + 127) // 128 for s in seq)
    table = np.zeros((nreq, width), np.int32)
    perm = rng.permutation(nb)
    k = 0
    for r in range(nreq):
        n = (seq[r] + 127) // 128
        table[r, :n] = perm[k:k + n]
        k += n
    kc = workloads.attend_kv_pages(seed, 0, np.arange(nb), H)
    vc = workloads.attend_kv_pages(seed, 1, np.arange(nb), H)
    req = np.array([0, 0, 1, 1, 1], np.int32)
    pos = np.array([seq[0] - 2, seq[0] - 1, seq[1] - 3, 130, 5], np.int32)
    T = req.size
    ids = np.full((T, H, 16), -1, np.int32)
    for t in range(T):
        L = pos[t] // 128
        for h in range(H):
            hist = rng.permutation(L)[:min(15, L)] if L else np.zeros(0, int)
            ids[t, h, :hist.size] = hist
            ids[t, h, hist.size] = L
    q = workloads.attend_q(T, H * G, rng)
    return q, kc, vc, table, req, pos, ids, G


def pin_brute_force():
    q, kc, vc, table, req, pos, ids, G = _case(1)
    scale = 128 ** -0.5
    o, _ = oat.attend(q, kc, vc, table, req, pos, ids, G, scale)
    for t in range(q.shape[0]):
        for hq in range(q.shape[1]):
            want = brute.attend_one(q[t, hq], kc, vc, table[req[t]], int(pos[t]), ids[t, hq // G], hq // G, scale)
            if np.max(np.abs(o[t, hq] - np.array(want))) > 1e-12:
                return f"row {t} head {hq}: differs from the brute force"
    return None


def pin_one_visible_token_is_its_v():
    q, kc, vc, table, req, pos, ids, G = _case(2)
    ids[:] = -1
    pos[:] = 128 * 2                               # local page 2, first token only
    ids[:, :, 0] = 2
    o, n = oat.attend(q, kc, vc, table, req, pos, ids, G, 0.3)
    for t in range(q.shape[0]):
        for hq in range(q.shape[1]):
            v = oat.bf16_value(vc[table[req[t], 2], 0, hq // G])
            if n[t, hq] != 1 or not np.array_equal(o[t, hq], v):
                return f"row {t} head {hq}: one visible token should give its v row"
    return None


def pin_zero_query_is_mean():
    q, kc, vc, table, req, pos, ids, G = _case(3)
    q[:] = 0
    o, _ = oat.attend(q, kc, vc, table, req, pos, ids, G, 0.3)
    for t in range(q.shape[0]):
        for hq in range(q.shape[1]):
            hk = hq // G
            rows = [oat.bf16_value(vc[table[req[t], j], s, hk])
                    for j in ids[t, hk] if j >= 0 for s in range(128) if 128 * j + s <= pos[t]]
            if np.max(np.abs(o[t, hq] - np.mean(rows, axis=0))) > 1e-12:
                return f"row {t} head {hq}: zero query should average the visible v rows"
    return None


def pin_causal_cut_and_empty_rows():
    """The local page is cut after the row's position: tokens past it never
    count (changing their K / V changes nothing, changing the last visible
    one does); all -1 gives zeros."""
    q, kc, vc, table, req, pos, ids, G = _case(4)
    for t in range(q.shape[0]):
        sl = slice(t, t + 1)
        o, _ = oat.attend(q[sl], kc, vc, table, req[sl], pos[sl], ids[sl], G, 0.3)
        blk, last = table[req[t], pos[t] // 128], pos[t] % 128
        kc2, vc2 = kc.copy(), vc.copy()
        kc2[blk, last + 1:] ^= 0x1234
        vc2[blk, last + 1:] ^= 0x4321
        o2, _ = oat.attend(q[sl], kc2, vc2, table, req[sl], pos[sl], ids[sl], G, 0.3)
        if not np.array_equal(o, o2):
            return f"row {t}: tokens after the row's position changed its output"
        vc2[blk, last] ^= 0x4321
        o3, _ = oat.attend(q[sl], kc2, vc2, table, req[sl], pos[sl], ids[sl], G, 0.3)
        if np.array_equal(o, o3):
            return f"row {t}: the token at the row's position is not seen"
    ids[:] = -1
    o3, n3 = oat.attend(q, kc, vc, table, req, pos, ids, G, 0.3)
    if np.any(o3 != 0) or np.any(n3 != 0):
        return "a row with no selected page should give zeros"
    return None


def pin_id_order_and_skips():
    q, kc, vc, table, req, pos, ids, G = _case(5)
    o, _ = oat.attend(q, kc, vc, table, req, pos, ids, G, 0.3)
    rng = np.random.Generator(np.random.PCG64(6))
    ids2 = ids.copy()
    for t in range(ids.shape[0]):
        for h in range(ids.shape[1]):
            ids2[t, h] = ids[t, h][rng.permutation(16)]      # -1 entries land anywhere
    o2, _ = oat.attend(q, kc, vc, table, req, pos, ids2, G, 0.3)
    if np.max(np.abs(o - o2)) > 1e-12:
        return "the order of the ids (and the place of the -1 entries) changed the output"
    return None


def pin_repeated_id_counts_once():
    """The visible set is a union of pages: an id listed twice for a row
    gives the brute force's answer over the set of pages, and the same
    output as the list with the repeat replaced by -1."""
    q, kc, vc, table, req, pos, ids, G = _case(8)
    scale = 128 ** -0.5
    ids2 = ids.copy()
    for t in range(ids.shape[0]):
        for h in range(ids.shape[1]):
            row = ids[t, h]
            valid = row[row >= 0]
            if valid.size >= 2 and (row < 0).any():
                ids2[t, h, np.nonzero(row < 0)[0][0]] = valid[valid.size // 2]   # a repeat in a free slot
    if np.array_equal(ids2, ids):
        return "the case has no row with a free slot for a repeated id"
    o, _ = oat.attend(q, kc, vc, table, req, pos, ids, G, scale)
    o2, _ = oat.attend(q, kc, vc, table, req, pos, ids2, G, scale)
    if np.max(np.abs(o - o2)) > 1e-12:
        return "a repeated id changed the output"
    t, hq = 0, 0
    want = brute.attend_one(q[t, hq], kc, vc, table[req[t]], int(pos[t]), ids2[t, hq // G], hq // G, scale)
    if np.max(np.abs(o2[t, hq] - np.array(want))) > 1e-12:
        return "a row with a repeated id differs from the brute force"
    return None


def _fp32_online(q, kc, vc, table, req, pos, ids, G, scale):
    """fp32 evaluation the way a kernel does it: page by page (ids order),
    per page the scores, a running max, rescaling of the accumulators, sums
    of at most 128 terms per page."""
    T, HQ, _ = q.shape
    out = np.zeros((T, HQ, 128), np.float32)
    f = lambda b: oat.bf16_value(b).astype(np.float32)
    for t in range(T):
        for hq in range(HQ):
            hk = hq // G
            m, l, acc = np.float32(-np.inf), np.float32(0), np.zeros(128, np.float32)
            qq = f(q[t, hq])
            for j in ids[t, hk]:
                if j < 0 or 128 * j > pos[t]:
                    continue
                n = min(128, int(pos[t]) - 128 * int(j) + 1)
                blk = table[req[t], j]
                K, V = f(kc[blk, :n, hk]), f(vc[blk, :n, hk])
                s = (K @ qq) * np.float32(scale)
                mn = max(m, s.max())
                a = np.exp(np.float32(m - mn)) if np.isfinite(m) else np.float32(0)
                p = np.exp((s - mn).astype(np.float32))
                l = l * a + p.sum(dtype=np.float32)
                acc = acc * a + (p @ V).astype(np.float32)
                m = mn
            if l > 0:
                out[t, hq] = acc / l
    return out


def pin_fp32_bound_covers_and_detects_a_dropped_token():
    q, kc, vc, table, req, pos, ids, G = _case(7, seq=(1500, 2100), nb=32)
    scale = 128 ** -0.5
    o, _ = oat.attend(q, kc, vc, table, req, pos, ids, G, scale)
    b = oat.error_bound(q, kc, vc, table, req, pos, ids, G, scale, chain=128)
    o32 = _fp32_online(q, kc, vc, table, req, pos, ids, G, scale).astype(np.float64)
    if np.any(np.abs(o32 - o) > b):
        return "an fp32 evaluation lies outside the error bound"
    # one token fewer: row 0 without the token at its own position
    pos2 = pos.copy()
    pos2[0] -= 1
    o_drop, _ = oat.attend(q, kc, vc, table, req, pos2, ids, G, scale)
    if not np.all(np.any(np.abs(o_drop[0] - o[0]) > b[0], axis=1)):
        return "removing one visible token stays inside the bound (bound too loose)"
    return None


PINS = [pin_brute_force, pin_one_visible_token_is_its_v, pin_zero_query_is_mean, pin_causal_cut_and_empty_rows,
        pin_id_order_and_skips, pin_repeated_id_counts_once, pin_fp32_bound_covers_and_detects_a_dropped_token]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin() is None


# ---------------------------------------------------------------- planted mistakes
_orig_visible = oat.visible_tokens
_orig_attend = oat.attend


def _visible_off_by_one(ids_row, table_row, pos):
    return _orig_visible(ids_row, table_row, pos - 1)


def _visible_logical_as_physical(ids_row, table_row, pos):
    return _orig_visible(ids_row, np.arange(len(table_row)), pos)


def _visible_first_id_skipped(ids_row, table_row, pos):
    r = np.array(ids_row).copy()
    r[0] = -1
    return _orig_visible(r, table_row, pos)


def _visible_repeats_counted(ids_row, table_row, pos):
    # every listed id read, a repeated one twice (a multiset instead of the union)
    b, s = [], []
    for j in np.asarray(ids_row).tolist():
        if j < 0:
            continue
        bb, ss = _orig_visible(np.array([j]), table_row, pos)
        b.append(bb)
        s.append(ss)
    if not b:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(b), np.concatenate(s)


def _attend_no_scale(q, kc, vc, table, req, pos, ids, G, scale):
    return _orig_attend(q, kc, vc, table, req, pos, ids, G, 1.0)


def _attend_wrong_head_group(q, kc, vc, table, req, pos, ids, G, scale):
    # query head hq read with KV head hq % H instead of hq // G
    T, HQ, _ = q.shape
    H = HQ // G
    q2 = q.reshape(T, H, G, 128).transpose(0, 2, 1, 3).reshape(T, HQ, 128)
    return _orig_attend(q2, kc, vc, table, req, pos, ids, G, scale)


MUTATIONS = [
    ("causal cut one token early", "visible_tokens", _visible_off_by_one,
     ["pin_brute_force", "pin_one_visible_token_is_its_v"]),
    ("logical page used as the physical block", "visible_tokens", _visible_logical_as_physical,
     ["pin_brute_force", "pin_one_visible_token_is_its_v"]),
    ("first id skipped", "visible_tokens", _visible_first_id_skipped,
     ["pin_brute_force", "pin_one_visible_token_is_its_v"]),
    ("repeated id counted twice", "visible_tokens", _visible_repeats_counted, ["pin_repeated_id_counts_once"]),
    ("scale ignored", "attend", _attend_no_scale, ["pin_brute_force"]),
    ("query head grouped with the wrong KV head", "attend", _attend_wrong_head_group, ["pin_brute_force"]),
]


def _fails(pin):
    try:
        return pin() is not None
    except Exception:
        return True


@pytest.mark.parametrize("name,attr,bad,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, attr, bad, pins):
    by_name = {p.__name__: p for p in PINS}
    for n in pins:
        assert by_name[n]() is None, n
    monkeypatch.setattr(oat, attr, bad)
    assert any(_fails(by_name[n]) for n in pins), f"planted mistake not caught: {name}"
