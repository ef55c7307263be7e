"""Fused qk-norm + RoPE + NVFP4 insert (nvfp4_insert_norm_rope) against the
oracle (oracle/norm_rope.py + oracle/nvfp4.py): every written row equals
the NVFP4 quantisation of the float64 qk-norm + RoPE key rounded to bf16,
except where an element of the key lies within the fp32 error bound of a
bf16 rounding boundary, where the row of the other neighbour is accepted
too (``norm_rope.check_rows``; the number of rows that needed it is
printed).  Rows of skipped tokens keep the cache's old bytes."""
import numpy as np
import pytest

import workloads
from oracle import norm_rope as onr
from gpu_util import torch_dev, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def rope_table(max_pos, rotary_dim, base=10000.0):
    """cos / sin table [max_pos, rotary_dim] of the standard RoPE frequencies
    base^(-2i / rotary_dim), cosines first (an input of the insert)."""
    h = rotary_dim // 2
    inv = base ** (-np.arange(h, dtype=np.float64) * 2.0 / rotary_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def case(n, seed, max_pos=4096):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x *= np.exp2(rng.integers(-6, 7, size=(n, 1))).astype(np.float32)     # spread of key norms
    x[:, rng.integers(0, 128, 4)] *= 8.0                                   # outlier channels
    k = workloads._to_bf16_bits(x)
    w = workloads._to_bf16_bits(rng.uniform(0.25, 2.0, 128).astype(np.float32))
    pos = rng.integers(0, max_pos, n).astype(np.int64)
    return k, w, pos


def assert_rows(got, k, pos, slots, w, eps, table, rd, neox, fill, label):
    """Rows written for the kept tokens pass the oracle's row check; every
    other row still holds ``fill``."""
    keep = onr.kept_tokens(pos, slots, table, rd)
    flat = got.reshape(-1, 72)
    rep = onr.check_rows(flat[slots[keep]], k[keep], pos[keep], w, eps, table, rd, neox)
    print(f"{label}: {rep['rows']} rows, {rep['exact']} exact, {rep['allowance']} within the bf16 "
          f"boundary allowance, {rep['fails']} failed {rep['fail_rows']}")
    assert rep["fails"] == 0, rep
    assert rep["allowance"] <= max(2, rep["rows"] // 1000), rep
    untouched = np.ones(flat.shape[0], bool)
    untouched[slots[keep]] = False
    assert np.all(flat[untouched] == fill)
    return rep


def run_gpu(k, pos, slots, w, eps, table, rd, neox, nb, fill=0):
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    kv = torch.full((nb, 128, 72), fill, dtype=torch.uint8, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    idx.insert_norm_rope(up(k.view(np.int16)), up(pos), up(slots), up(w.view(np.int16)), eps,
                         up(table) if table is not None else None, rd, neox, kv, status=status)
    return kv.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("rd,neox", [(128, True), (64, True), (128, False), (64, False), (40, False),
                                     (32, False), (6, False), (2, False), (0, True)])
def test_norm_rope_insert_matches_oracle(rd, neox):
    n = 20000
    k, w, pos = case(n, 40 + rd + neox)
    nb = (n + 127) // 128 + 3
    rng = np.random.Generator(np.random.PCG64(41))
    slots = rng.permutation(nb * 128)[:n].astype(np.int64)
    slots[::11] = -1
    table = rope_table(4096, rd) if rd else None
    got, st = run_gpu(k, pos, slots, w, 1e-6, table, rd, neox, nb, fill=0x5A)
    assert st == 0
    assert_rows(got, k, pos, slots, w, 1e-6, table, rd, neox, 0x5A, f"rd {rd} neox {neox}")


@pytest.mark.parametrize("rd,neox", [(64, True), (128, False), (6, False), (0, True)])
def test_norm_rope_insert_many_blocks(rd, neox):
    """Some 49 000 keys (many blocks of 64 tokens and a ragged last one),
    skipped slots and positions past the table: 4096 sampled kept rows
    checked against the oracle, every other row of the cache untouched."""
    n = 152 * 32 * 10 + 19
    k, w, pos = case(n, 60 + rd + neox, max_pos=2048)
    nb = (n + 127) // 128 + 2
    rng = np.random.Generator(np.random.PCG64(61))
    slots = rng.permutation(nb * 128)[:n].astype(np.int64)
    slots[::13] = -1
    table = rope_table(2000, rd) if rd else None
    got, st = run_gpu(k, pos, slots, w, 1e-6, table, rd, neox, nb, fill=0x33)
    import sparse_attention_block_nvfp4_gb300 as idx
    assert st == (idx.STATUS_BAD_POSITION if rd else 0)
    keep = onr.kept_tokens(pos, slots, table, rd)
    assert 0.9 * n < keep.sum() < n
    flat = got.reshape(-1, 72)
    untouched = np.ones(flat.shape[0], bool)
    untouched[slots[keep]] = False
    assert np.all(flat[untouched] == 0x33)
    pick = rng.choice(np.nonzero(keep)[0], size=4096, replace=False)
    rep = onr.check_rows(flat[slots[pick]], k[pick], pos[pick], w, 1e-6, table, rd, neox)
    print(f"rd {rd} neox {neox}, 4096 sampled rows: {rep}")
    assert rep["fails"] == 0, rep
    assert rep["allowance"] <= 4, rep


def test_norm_rope_insert_eps_and_extremes():
    """Large eps against small keys, zero keys, keys near bf16's range edges,
    a weight with zeros and negatives: still within the oracle's check."""
    rng = np.random.Generator(np.random.PCG64(42))
    n = 512
    x = rng.standard_normal((n, 128)).astype(np.float32)
    x[:64] *= 1e-3
    x[64:128] = 0.0
    x[128:192] *= np.float32(2.0 ** 60)
    x[192:256] *= np.float32(2.0 ** -60)
    k = workloads._to_bf16_bits(x)
    wv = rng.uniform(-2.0, 2.0, 128).astype(np.float32)
    wv[::9] = 0.0
    w = workloads._to_bf16_bits(wv)
    pos = rng.integers(0, 300, n).astype(np.int64)
    table = rope_table(300, 128)
    slots = np.arange(n, dtype=np.int64)
    for eps in (1e-6, 0.5):
        got, st = run_gpu(k, pos, slots, w, eps, table, 128, True, 4)
        assert st == 0
        assert_rows(got, k, pos, slots, w, eps, table, 128, True, 0, f"eps {eps}")


def test_norm_rope_insert_bad_positions_and_slots():
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    k, w, pos = case(8, 43, max_pos=64)
    pos[2] = 64                                   # past the table
    pos[5] = -3
    slots = np.arange(8, dtype=np.int64)
    slots[6] = 10 * 128                           # past the cache
    table = rope_table(64, 128)
    got, st = run_gpu(k, pos, slots, w, 1e-6, table, 128, True, 1, fill=0x77)
    assert st == idx.STATUS_BAD_POSITION | idx.STATUS_BAD_SLOT
    ok = np.array([0, 1, 3, 4, 7])
    assert np.array_equal(np.nonzero(onr.kept_tokens(pos, np.where(slots < 128, slots, -1), table, 128))[0], ok)
    assert_rows(got, k[ok], pos[ok], slots[ok], w, 1e-6, table, 128, True, 0x77, "bad positions and slots")
    with pytest.raises(idx.IndexerError) as e:
        run_gpu(k, pos, slots, w, 1e-6, rope_table(64, 96), 96, True, 1)
    assert e.value.code == idx.IDX_EUNSUPPORTED
    with pytest.raises(idx.IndexerError):
        run_gpu(k, pos, slots, w, -1.0, table, 128, True, 1)


@pytest.mark.parametrize("rd,neox", [(128, True), (64, True), (40, False), (6, False), (0, True)])
def test_norm_rope_insert_keys_16_byte_aligned(rd, neox):
    """Keys at an address that is 16-byte but not 32-byte aligned (the
    kernel then loads each group in two 16-byte halves instead of one
    32-byte load): the same rows as from 32-byte aligned keys, and within
    the oracle's check."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    n = 3000
    k, w, pos = case(n, 90 + rd + neox)
    nb = (n + 127) // 128 + 1
    slots = np.arange(n, dtype=np.int64)[::-1].copy()
    slots[::7] = -1
    table = rope_table(4096, rd) if rd else None
    outs = []
    for off in (0, 8):                            # int16 elements: 0 or 16 bytes
        buf = torch.zeros(n * 128 + 16, dtype=torch.int16, device=torch_dev())
        kd = buf[off:off + n * 128].view(n, 128)
        kd.copy_(up(k.view(np.int16)))
        assert (kd.data_ptr() % 32 == 0) == (off == 0) and kd.data_ptr() % 16 == 0
        kv = torch.full((nb, 128, 72), 0x21, dtype=torch.uint8, device=torch_dev())
        status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
        idx.insert_norm_rope(kd, up(pos), up(slots), up(w.view(np.int16)), 1e-6,
                             up(table) if table is not None else None, rd, neox, kv, status=status)
        assert int(status.item()) == 0
        outs.append(kv.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    assert_rows(outs[1], k, pos, slots, w, 1e-6, table, rd, neox, 0x21, f"16-byte aligned keys, rd {rd}")


def test_norm_rope_insert_full_cache_sampled():
    """The long mixed workload's whole cache (2.24 M keys, each request's
    tokens at positions 0 .. seq_len - 1), in the launch configuration the
    benchmark times; 16384 sampled rows checked against the oracle."""
    w_ = workloads.config(4)
    seq = np.concatenate([w_.dec_seq_lens, w_.pre_seq_lens]).astype(np.int64)
    pos = np.concatenate([np.arange(s) for s in seq])
    assert pos.size == w_.k_bf16.shape[0]
    rng = np.random.Generator(np.random.PCG64(44))
    wts = workloads._to_bf16_bits(rng.uniform(0.5, 1.5, 128).astype(np.float32))
    table = rope_table(int(seq.max()), 128)
    got, st = run_gpu(w_.k_bf16, pos, w_.slot_mapping, wts, 1e-6, table, 128, True, w_.num_blocks)
    assert st == 0
    pick = rng.choice(pos.size, size=16384, replace=False)
    rep = onr.check_rows(got.reshape(-1, 72)[w_.slot_mapping[pick]], w_.k_bf16[pick], pos[pick], wts, 1e-6,
                         table, 128, True)
    print(f"full cache, 16384 sampled rows: {rep}")
    assert rep["fails"] == 0, rep
    assert rep["allowance"] <= 16, rep
