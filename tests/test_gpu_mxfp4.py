"""MXFP4 pages on the GPU (mxfp4_insert, indexer_decode_mxfp4,
indexer_prefill_mxfp4) against the CPU oracle: insert bytes bit-exact, ids
and scores within the checker's tolerance."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import indexer as oidx
from oracle import mxfp4 as omx
from gpu_util import assert_ids, assert_scores, make_plan, torch_dev, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def gpu_mx_cache(w):
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    pages = torch.zeros((w.num_blocks, omx.PAGE_BYTES), dtype=torch.uint8, device=torch_dev())
    idx.mxfp4_insert(up(w.k_bf16.view(np.int16)), up(w.slot_mapping), pages)
    return pages


def oracle_mx_cache(w):
    return omx.insert(w.k_bf16, w.slot_mapping, np.zeros((w.num_blocks, omx.PAGE_BYTES), np.uint8))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_mxfp4_insert_bit_exact_small_workloads(idx):
    w = workloads.config(idx, small=True)
    got = gpu_mx_cache(w).cpu().numpy()
    want = oracle_mx_cache(w)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"


def test_mxfp4_insert_edge_values():
    """The hand-worked block, blocks spread over every binade (subnormal
    amax, clamped exponents, saturation), signed zeros, arbitrary finite bf16
    patterns; negative slots skipped, out-of-range slots flagged."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_quantize.json")))
    row = np.zeros(128, np.uint16)
    for k, v in g["x_bf16_nonzero"].items():
        row[int(k)] = int(v, 16)
    rng = np.random.Generator(np.random.PCG64(31))
    rows = [row]
    pat = rng.integers(0, 1 << 16, size=(200, 128), dtype=np.uint32).astype(np.uint16)
    pat[(pat & 0x7F80) == 0x7F80] &= 0xBF7F          # no inf / NaN
    rows.append(pat)
    mant = rng.standard_normal((100, 128)).astype(np.float32)
    spread = np.exp2(rng.integers(-140, 126, size=(100, 4)).astype(np.float32))
    x = (mant * np.repeat(spread, 32, axis=1)).view(np.uint32)
    rows.append(((x + 0x7FFF + ((x >> 16) & 1)) >> 16).astype(np.uint16))
    z = np.zeros((2, 128), np.uint16)
    z[1, ::3] = 0x8000                                 # -0.0
    rows.append(z)
    k = np.concatenate([np.atleast_2d(r) for r in rows]).astype(np.uint16)
    n = k.shape[0]
    nb = (n + 127) // 128 + 1
    slots = rng.permutation(nb * 128)[:n].astype(np.int64)
    slots[::17] = -1
    want = omx.insert(k, slots, np.zeros((nb, omx.PAGE_BYTES), np.uint8))
    pages = torch.zeros((nb, omx.PAGE_BYTES), dtype=torch.uint8, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    idx.mxfp4_insert(up(k.view(np.int16)), up(slots), pages, status=status)
    got = pages.cpu().numpy()
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"
    assert int(status.item()) == 0
    bad = np.array([nb * 128 + 5], np.int64)
    idx.mxfp4_insert(up(k[:1].view(np.int16)), up(bad), pages, status=status)
    assert int(status.item()) == 8                      # IDX_STATUS_BAD_SLOT
    assert np.array_equal(pages.cpu().numpy(), want)


def _every_value_every_exponent():
    """Blocks that pair every finite bf16 value with every shared exponent
    it can meet: for each biased exponent field e of amax (1 .. 254) the
    block's element 0 is the largest bf16 with that field (E = e - 129,
    clamped to -127) and the other 31 run over every x with |x| <= amax."""
    from oracle.formats import bf16_value
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    mag = np.abs(bf16_value(bits))
    order = np.argsort(mag, kind="stable")
    bits, mag = bits[order], mag[order]
    blocks = []
    for e in range(1, 255):
        amax_bits = np.uint16((e << 7) | 0x7F)
        amax = bf16_value(np.array([amax_bits]))[0]
        xs = bits[:np.searchsorted(mag, amax, side="right")]
        xs = np.concatenate([xs, np.zeros((-xs.size) % 31, np.uint16)]).reshape(-1, 31)
        blocks.append(np.concatenate([np.full((xs.shape[0], 1), amax_bits, np.uint16), xs], 1))
    g = np.concatenate(blocks)
    g = np.concatenate([g, np.zeros(((-g.shape[0]) % 4, 32), np.uint16)])
    return g.reshape(-1, 128)


def test_mxfp4_insert_exhaustive_bit_exact():
    """Every finite bf16 key value against every shared exponent: the
    kernel's bytes equal the oracle's exact rounding."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    k = _every_value_every_exponent()
    n = k.shape[0]
    nb = (n + 127) // 128
    slots = np.arange(n, dtype=np.int64)
    pages = torch.zeros((nb, omx.PAGE_BYTES), dtype=torch.uint8, device=torch_dev())
    idx.mxfp4_insert(up(k.view(np.int16)), up(slots), pages)
    want = omx.insert(k, slots, np.zeros((nb, omx.PAGE_BYTES), np.uint8))
    got = pages.cpu().numpy()
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"


def _run_decode(plan, w, pages, dbg=True):
    import torch
    d = torch.full((w.num_decode_rows, w.num_heads, w.page_table.shape[1]), float("nan"),
                   dtype=torch.float32, device=torch_dev()) if dbg else None
    out = plan.decode_mxfp4(up(w.q_decode), pages, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len,
                            scores_dbg=d)
    return out.cpu().numpy(), (d.cpu().numpy() if dbg else None)


def _run_prefill(plan, w, pages, dbg=True):
    import torch
    d = torch.full((w.total_prefill_q, w.num_heads, w.page_table.shape[1]), float("nan"),
                   dtype=torch.float32, device=torch_dev()) if dbg else None
    out = plan.prefill_mxfp4(up(w.q_prefill), up(w.cu_seqlens_q), pages, up(w.pre_page_table),
                             up(w.pre_seq_lens), int(w.pre_query_lens.max()), scores_dbg=d)
    return out.cpu().numpy(), (d.cpu().numpy() if dbg else None)


def _check_decode(w):
    pages = gpu_mx_cache(w)
    plan = make_plan(w)
    out, sc = _run_decode(plan, w, pages)
    ref = oidx.decode(w.q_decode, oracle_mx_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len,
                      w.num_heads, page_format="mxfp4")
    assert_ids(out, ref, w.name)
    assert_scores(sc, ref, w.name)
    assert plan.status() == 0
    plan.close()


def _check_prefill(w):
    pages = gpu_mx_cache(w)
    plan = make_plan(w)
    out, sc = _run_prefill(plan, w, pages)
    ref = oidx.prefill(w.q_prefill, w.cu_seqlens_q, oracle_mx_cache(w), w.pre_page_table, w.pre_seq_lens,
                       w.num_heads, page_format="mxfp4")
    assert_ids(out, ref, w.name)
    assert_scores(sc, ref, w.name)
    assert plan.status() == 0
    plan.close()


@pytest.mark.parametrize("idx", [0, 1, 2, 4])
def test_mxfp4_decode_parity_small_workloads(idx):
    _check_decode(workloads.config(idx, small=True))


@pytest.mark.parametrize("H,qlen", [(1, 1), (2, 3), (8, 8)])
def test_mxfp4_decode_heads_and_query_lens(H, qlen):
    rng = np.random.Generator(np.random.PCG64(80 + H))
    seq = [qlen - 1, 128 * 3 + 1, 2000, 128 * 17, 5000]
    w = workloads.make_workload(name=f"mxdec_H{H}", seed=80 + H, rng=rng, num_heads=H,
                                dec_seq_lens=seq, query_len=qlen, outlier_channels=4,
                                page_scale_spread=6.0)
    _check_decode(w)


@pytest.mark.parametrize("idx", [3, 4])
def test_mxfp4_prefill_parity_small_workloads(idx):
    _check_prefill(workloads.config(idx, small=True))


@pytest.mark.parametrize("H", [1, 8])
def test_mxfp4_prefill_heads_ragged_and_cut_units(H):
    rng = np.random.Generator(np.random.PCG64(90 + H))
    ctx = [0, 0, 300, 128 * 9, 5, 128 * 40, 127]
    new = [1, 129, 77, 530, 300, 700, 1]
    seq = [c + n for c, n in zip(ctx, new)]
    w = workloads.make_workload(name=f"mxpre_H{H}", seed=90 + H, rng=rng, num_heads=H,
                                pre_seq_lens=seq, pre_query_lens=new, outlier_channels=4,
                                page_scale_spread=6.0)
    _check_prefill(w)
