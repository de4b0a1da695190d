"""Pins of the oracle against what the pages and the mathematics fix.

Both oracle implementations (numpy ``reference`` and C ``native``) are held to
the same pins:
  * the pages' worked examples (block counts, tail slots, table lookups);
  * attention on an identity layout equals a library routine
    (``torch.nn.functional.scaled_dot_product_attention`` in float64);
  * closed forms: one token -> its value row; equal keys -> mean of values;
    one dominant score -> that token's value row; no token -> zeros;
  * invariants: relabelling physical blocks, shared vs privately copied
    layouts, and unused pool content do not change the result;
  * write / copy: bit-exact against a library reshape of the pool.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conftest import read_golden
from oracle import native, reference

IMPLS = {"numpy": reference, "c": native}


@pytest.fixture(params=sorted(IMPLS), scope="module")
def orc(request):
    return IMPLS[request.param]


# --------------------------------------------------------------- worked examples
def test_block_layout_golden(orc):
    for tokens, bs, blocks, unused in read_golden("block_layout.txt"):
        assert orc.block_layout(int(tokens), int(bs)) == (int(blocks), int(unused))


def test_block_layout_tail_bound(orc):
    # For every n < 100 at block size 4: blocks * 4 >= n and 0 <= unused < 4.
    for n in range(100):
        b, unused = orc.block_layout(n, 4)
        assert b * 4 >= n and 0 <= unused < 4
        assert b * 4 - unused == n
        assert (b == 0) == (n == 0)


def test_block_layout_rejects_invalid(orc):
    for tokens, bs in [(-1, 4), (5, 0), (5, -3)]:
        with pytest.raises(ValueError):
            orc.block_layout(tokens, bs)


def test_lookup_golden(orc):
    for table, bs, pos, phys, off in read_golden("block_lookup.txt"):
        row = [int(x) for x in table.split(",")]
        assert orc.locate(row, int(pos), int(bs)) == (int(phys), int(off))


def test_slot_of_golden():
    # [5, 1, 7], B = 4, position 9 -> physical 7, offset 1 -> flat slot 29
    for impl in (reference, native):
        assert list(impl.slot_mapping([[5, 1, 7]], [0], [9], 4)) == [29]


def test_lookup_past_table_raises(orc):
    with pytest.raises(IndexError):
        orc.locate([5, 1, 7], 12, 4)


# --------------------------------------------------------------- decode helpers
def _identity_case(S, Hq, Hkv, D, B, blocks_per_seq, dtype=torch.float64, seed=0):
    """Pool whose table for sequence s is the contiguous run s*n .. s*n+n-1."""
    g = torch.Generator().manual_seed(seed)
    NB = S * blocks_per_seq
    k = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    v = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    tables = np.arange(NB, dtype=np.int32).reshape(S, blocks_per_seq)
    return q, k, v, tables


def _sdpa_reference(q, k, v, lens, scale):
    """Library routine on contiguous K/V: sequence s's tokens are the rows of its
    blocks in table order, here read off the pool with a reshape."""
    S, Hq, D = q.shape
    NB, Hkv, B, _ = k.shape
    n = NB // S
    out = torch.zeros(S, Hq, D, dtype=torch.float64)
    for s in range(S):
        L = int(lens[s])
        if L == 0:
            continue
        # [n][Hkv][B][D] -> [Hkv][n*B][D]: contiguous history per KV head
        Ks = k[s * n:(s + 1) * n].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, n * B, D)[:, :L]
        Vs = v[s * n:(s + 1) * n].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, n * B, D)[:, :L]
        Ks = Ks.repeat_interleave(Hq // Hkv, dim=0)  # query head h reads KV head h // G
        Vs = Vs.repeat_interleave(Hq // Hkv, dim=0)
        qs = q[s].to(torch.float64).unsqueeze(1)   # [Hq][1][D]
        out[s] = F.scaled_dot_product_attention(qs, Ks, Vs, scale=scale).squeeze(1)
    return out.numpy()


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 3)])
def test_decode_identity_layout_matches_sdpa(orc, Hq, Hkv):
    S, D, B, n = 3, 16, 4, 5
    q, k, v, tables = _identity_case(S, Hq, Hkv, D, B, n, dtype=torch.float32, seed=Hq)
    lens = np.array([17, 20, 1], dtype=np.int32)   # ragged tail, full, single token
    scale = 0.37
    got = orc.decode(q, k, v, tables, lens, scale)
    want = _sdpa_reference(q, k, v, lens, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def _random_paged(S, Hq, Hkv, D, B, NB, lens, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    v = torch.randn(NB, Hkv, B, D, generator=g).to(dtype)
    q = torch.randn(S, Hq, D, generator=g).to(dtype)
    width = max(-(-int(L) // B) for L in lens) if len(lens) else 0
    perm = torch.randperm(NB, generator=g)[: S * width].view(S, width).numpy().astype(np.int32)
    return q, k, v, perm


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_decode_invariant_under_block_relabelling(orc, dtype):
    S, Hq, Hkv, D, B, NB = 3, 4, 2, 32, 4, 40
    lens = np.array([13, 4, 30], dtype=np.int32)
    q, k, v, tables = _random_paged(S, Hq, Hkv, D, B, NB, lens, dtype, seed=3)
    base = orc.decode(q, k, v, tables, lens, 0.2)
    pi = torch.randperm(NB, generator=torch.Generator().manual_seed(11))
    k2 = torch.empty_like(k)
    v2 = torch.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    tables2 = pi.numpy().astype(np.int32)[tables]
    again = orc.decode(q, k2, v2, tables2, lens, 0.2)
    assert np.array_equal(base, again)
    # unused blocks and slots past each context do not matter
    used = set(tables.ravel().tolist())
    k3, v3 = k.clone(), v.clone()
    for p in range(NB):
        if p not in used:
            k3[p] = 1e4
            v3[p] = -1e4
    assert np.array_equal(base, orc.decode(q, k3, v3, tables, lens, 0.2))


def test_decode_shared_equals_private_copy(orc):
    # Two sequences point at the same first blocks (a shared prefix); the same
    # history copied into private blocks gives the identical result.
    D, B, Hq, Hkv = 16, 4, 4, 2
    g = torch.Generator().manual_seed(5)
    NB = 20
    k = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    v = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    q = torch.randn(2, Hq, D, generator=g).to(torch.bfloat16)
    shared = np.array([[0, 1, 2, 3], [0, 1, 4, 5]], dtype=np.int32)
    lens = np.array([15, 14], dtype=np.int32)
    kp, vp = k.clone(), v.clone()
    kp[10:12] = k[0:2]
    vp[10:12] = v[0:2]
    private = np.array([[0, 1, 2, 3], [10, 11, 4, 5]], dtype=np.int32)
    assert np.array_equal(orc.decode(q, k, v, shared, lens, 0.25),
                          orc.decode(q, kp, vp, private, lens, 0.25))


def test_decode_closed_forms(orc):
    D, B, Hq, Hkv = 8, 4, 2, 1
    g = torch.Generator().manual_seed(9)
    NB = 6
    v = torch.randn(NB, Hkv, B, D, generator=g, dtype=torch.float64).to(torch.float32)
    k = torch.randn(NB, Hkv, B, D, generator=g, dtype=torch.float64).to(torch.float32)
    q = torch.randn(4, Hq, D, generator=g, dtype=torch.float64).to(torch.float32)
    tables = np.array([[3, 0], [1, 2], [4, 5], [2, 1]], dtype=np.int32)
    # seq 1: all keys equal -> uniform weights -> mean of its 7 value rows
    k[1] = 0.5
    k[2, :, :3] = 0.5
    # seq 2: the key at position 5 is aligned with every query head and large
    k[5, 0, 1] = 60.0 * q[2, 0] / q[2, 0].norm()
    q[2, 1] = q[2, 0]
    lens = np.array([1, 7, 6, 0], dtype=np.int32)
    out = orc.decode(q, k, v, tables, lens, 1.0)
    vd = v.to(torch.float64).numpy()
    # one cached token -> its value row, exactly
    assert np.array_equal(out[0, 0], vd[3, 0, 0]) and np.array_equal(out[0, 1], vd[3, 0, 0])
    rows = np.concatenate([vd[1, 0], vd[2, 0, :3]])
    np.testing.assert_allclose(out[1], np.broadcast_to(rows.mean(0), (Hq, D)), rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[2], np.broadcast_to(vd[5, 0, 1], (Hq, D)), rtol=0, atol=1e-12)
    assert np.all(out[3] == 0.0)   # no cached token -> zero row


def test_decode_gqa_group_mapping(orc):
    # Query heads 0..3 read KV head 0 and 4..7 read KV head 1: give the two KV
    # heads constant, different values and check which value each head returns.
    S, Hq, Hkv, D, B = 1, 8, 2, 8, 4
    k = torch.randn(2, Hkv, B, D, generator=torch.Generator().manual_seed(1))
    v = torch.zeros(2, Hkv, B, D)
    v[:, 0] = 1.0
    v[:, 1] = 2.0
    q = torch.randn(S, Hq, D, generator=torch.Generator().manual_seed(2))
    out = orc.decode(q, k, v, np.array([[1, 0]], dtype=np.int32), np.array([6], dtype=np.int32), 0.3)
    np.testing.assert_allclose(out[0, :4], 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[0, 4:], 2.0, rtol=0, atol=1e-15)


def test_decode_rejects_context_past_table(orc):
    q, k, v, tables = _identity_case(1, 2, 2, 8, 4, 2, dtype=torch.float32)
    with pytest.raises((ValueError, IndexError)):
        orc.decode(q, k, v, tables, np.array([9], dtype=np.int32), 1.0)


def test_numpy_and_c_oracles_agree():
    S, Hq, Hkv, D, B, NB = 4, 8, 2, 64, 16, 64
    lens = np.array([1, 17, 100, 64], dtype=np.int32)
    for dtype in (torch.float32, torch.float16, torch.bfloat16):
        q, k, v, tables = _random_paged(S, Hq, Hkv, D, B, NB, lens, dtype, seed=21)
        a = reference.decode(q, k, v, tables, lens, 1 / math.sqrt(D))
        b = native.decode(q, k, v, tables, lens, 1 / math.sqrt(D))
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- write / copy
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_write_kv_identity_slots(orc, dtype):
    # slots 0..T-1 fill the pool in order: read back with a library reshape
    NB, Hkv, B, D, T = 3, 2, 4, 8, 10
    g = torch.Generator().manual_seed(4)
    key = torch.randn(T, Hkv, D, generator=g).to(dtype)
    val = torch.randn(T, Hkv, D, generator=g).to(dtype)
    kc = torch.zeros(NB, Hkv, B, D, dtype=dtype)
    vc = torch.zeros(NB, Hkv, B, D, dtype=dtype)
    orc.write_kv(key, val, kc, vc, np.arange(T, dtype=np.int64))
    flat_k = kc.permute(0, 2, 1, 3).reshape(NB * B, Hkv, D)
    flat_v = vc.permute(0, 2, 1, 3).reshape(NB * B, Hkv, D)
    assert torch.equal(flat_k[:T], key) and torch.equal(flat_v[:T], val)
    assert torch.count_nonzero(flat_k[T:]) == 0 and torch.count_nonzero(flat_v[T:]) == 0


def test_write_kv_skips_negative_and_rejects_outside(orc):
    NB, Hkv, B, D = 2, 1, 4, 4
    kc = torch.zeros(NB, Hkv, B, D)
    vc = torch.zeros(NB, Hkv, B, D)
    key = torch.ones(2, Hkv, D)
    orc.write_kv(key, key, kc, vc, np.array([-1, 5], dtype=np.int64))
    assert torch.count_nonzero(kc) == D and torch.all(kc[1, 0, 1] == 1)
    with pytest.raises(IndexError):
        orc.write_kv(key, key, kc, vc, np.array([0, NB * B], dtype=np.int64))


def test_copy_blocks(orc):
    NB, Hkv, B, D = 6, 2, 4, 8
    g = torch.Generator().manual_seed(8)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    k0, v0 = kc.clone(), vc.clone()
    orc.copy_blocks(kc, vc, np.array([[1, 4], [2, 5]], dtype=np.int64))
    assert torch.equal(kc[4], k0[1]) and torch.equal(vc[5], v0[2])
    for p in (0, 1, 2, 3):
        assert torch.equal(kc[p], k0[p]) and torch.equal(vc[p], v0[p])
    # pairs apply in order: 0 -> 3 then 3 -> 1 leaves block 0's data in 1
    orc.copy_blocks(kc, vc, np.array([[0, 3], [3, 1]], dtype=np.int64))
    assert torch.equal(kc[1], k0[0]) and torch.equal(vc[3], v0[0])
    with pytest.raises(IndexError):
        orc.copy_blocks(kc, vc, np.array([[0, NB]], dtype=np.int64))


# ------------------------------------------------------------------ prefill
def _sdpa_prefill(q, k, v, lens, q_start, scale):
    """Library routine with an explicit causal mask on contiguous K/V: query row
    i of sequence s (position L - n + i) may see keys 0 .. L - n + i."""
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k.shape
    S = len(lens)
    nb = NB // S
    out = torch.zeros(T, Hq, D, dtype=torch.float64)
    for s in range(S):
        L, a, b = int(lens[s]), int(q_start[s]), int(q_start[s + 1])
        n = b - a
        if n == 0:
            continue
        Ks = k[s * nb:(s + 1) * nb].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :L]
        Vs = v[s * nb:(s + 1) * nb].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, nb * B, D)[:, :L]
        Ks = Ks.repeat_interleave(Hq // Hkv, dim=0)
        Vs = Vs.repeat_interleave(Hq // Hkv, dim=0)
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]   # [n][L], True = visible
        qs = q[a:b].to(torch.float64).transpose(0, 1)                             # [Hq][n][D]
        out[a:b] = F.scaled_dot_product_attention(qs, Ks, Vs, attn_mask=mask, scale=scale).transpose(0, 1)
    return out.numpy()


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2)])
def test_prefill_identity_layout_matches_sdpa(orc, Hq, Hkv):
    S, D, B, nb = 3, 16, 4, 6
    q_all, k, v, _ = _identity_case(S, Hq, Hkv, D, B, nb, dtype=torch.float32, seed=5 + Hq)
    tables = np.arange(S * nb, dtype=np.int32).reshape(S, nb)
    lens = np.array([17, 24, 5], dtype=np.int32)        # history + prompt
    q_start = np.array([0, 9, 9 + 24, 9 + 24 + 1], dtype=np.int32)  # prompts of 9, 24 (no history), 1
    q = torch.randn(int(q_start[-1]), Hq, D, generator=torch.Generator().manual_seed(Hq)).to(torch.float32)
    got = orc.prefill(q, k, v, tables, lens, q_start, 0.29)
    want = _sdpa_prefill(q, k, v, lens, q_start, 0.29)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_prefill_closed_forms(orc):
    # all keys equal: row i (position p) is the mean of V over 0 .. p
    S, Hq, Hkv, D, B, NB = 1, 2, 1, 8, 4, 3
    k = torch.zeros(NB, Hkv, B, D)
    v = torch.randn(NB, Hkv, B, D, generator=torch.Generator().manual_seed(2))
    tables = np.array([[2, 0, 1]], dtype=np.int32)
    L, n = 11, 4
    q = torch.randn(n, Hq, D, generator=torch.Generator().manual_seed(3))
    got = orc.prefill(q, k, v, tables, np.array([L], np.int32), np.array([0, n], np.int32), 1.0)
    rows = torch.cat([v[p, 0] for p in tables[0]])  # logical order [12][D]
    for i in range(n):
        p = L - n + i
        want = rows[:p + 1].double().mean(0).numpy()
        for h in range(Hq):
            np.testing.assert_allclose(got[i, h], want, rtol=1e-12, atol=1e-14)
    # a prompt of one token at position 0 returns its own value row
    got1 = orc.prefill(q[:1], k, v, tables, np.array([1], np.int32), np.array([0, 1], np.int32), 1.0)
    np.testing.assert_allclose(got1[0, 0], rows[0].double().numpy(), rtol=0, atol=0)


def test_prefill_last_row_is_the_decode_of_its_sequence(orc):
    S, Hq, Hkv, D, B, NB = 2, 4, 2, 16, 4, 24
    lens = np.array([14, 7], dtype=np.int32)
    qd, k, v, tables = _random_paged(S, Hq, Hkv, D, B, NB, lens, torch.float32, seed=8)
    q_start = np.array([0, 5, 12], dtype=np.int32)
    q = torch.randn(12, Hq, D, generator=torch.Generator().manual_seed(9))
    got = orc.prefill(q, k, v, tables, lens, q_start, 0.4)
    last = q[torch.as_tensor(q_start[1:] - 1, dtype=torch.long)]
    np.testing.assert_allclose(got[q_start[1:] - 1], orc.decode(last, k, v, tables, lens, 0.4), rtol=1e-12,
                               atol=1e-14)


def test_prefill_invariant_under_block_relabelling(orc):
    S, Hq, Hkv, D, B, NB = 2, 4, 2, 8, 4, 30
    lens = np.array([19, 9], dtype=np.int32)
    qd, k, v, tables = _random_paged(S, Hq, Hkv, D, B, NB, lens, torch.bfloat16, seed=12)
    q_start = np.array([0, 6, 15], dtype=np.int32)
    q = torch.randn(15, Hq, D, generator=torch.Generator().manual_seed(13)).to(torch.bfloat16)
    base = orc.prefill(q, k, v, tables, lens, q_start, 0.3)
    pi = torch.randperm(NB, generator=torch.Generator().manual_seed(14))
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    k2[pi], v2[pi] = k, v
    again = orc.prefill(q, k2, v2, pi.numpy().astype(np.int32)[tables], lens, q_start, 0.3)
    assert np.array_equal(base, again)


def test_prefill_implementations_agree_and_reject_bad_offsets():
    S, Hq, Hkv, D, B, NB = 3, 8, 2, 32, 16, 40
    lens = np.array([70, 33, 16], dtype=np.int32)
    _, k, v, tables = _random_paged(S, Hq, Hkv, D, B, NB, lens, torch.float16, seed=21)
    q_start = np.array([0, 20, 53, 54], dtype=np.int32)
    q = torch.randn(54, Hq, D, generator=torch.Generator().manual_seed(22)).to(torch.float16)
    a = reference.prefill(q, k, v, tables, lens, q_start, 0.18)
    b = native.prefill(q, k, v, tables, lens, q_start, 0.18)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):  # a prompt longer than its context
        native.prefill(q, k, v, tables, np.array([10, 33, 16], np.int32), q_start, 0.18)
