"""Pins for the fp64 oracle, checked against facts that do not come from it.

Each test fixes one part of the oracle against an independent source: a
library conversion, a brute-force search, a closed form, dense attention from
torch on contiguous copies, or an invariant of the definition (block-id
permutation, window = truncation).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


# ------------------------------------------------------------------ codecs

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def _e4m3_torch(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    ref = _e4m3_torch(codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_e4m3_decode_closed_forms():
    # OCP E4M3: largest finite 1.75 * 2^8, smallest normal 2^-6, smallest subnormal 2^-9
    v = oracle.e4m3_to_f64(np.array([0x7E, 0xFE, 0x08, 0x01, 0x38, 0xB8, 0x00, 0x80, 0x07],
                                    np.uint8))
    assert list(v[:6]) == [448.0, -448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0]
    assert v[6] == 0.0 and not np.signbit(v[6]) and v[7] == 0.0 and np.signbit(v[7])
    assert v[8] == 7 * 2.0 ** -9


def _finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def test_e4m3_encode_round_trips_every_finite_code():
    codes, vals = _finite_codes()
    enc = oracle.e4m3_from_f32(vals.astype(np.float32))
    assert (enc == codes).all()


def test_e4m3_encode_matches_torch_cast_below_overflow():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.normal(size=20000) * s for s in (1e-3, 0.01, 0.3, 1, 10, 100)
    ] + [rng.uniform(-463.9, 463.9, 20000), rng.uniform(-2 ** -6, 2 ** -6, 20000)])
    x = x.astype(np.float32)
    x = x[np.abs(x) < 464]
    got = oracle.e4m3_from_f32(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps -0 for negative values that round to zero, as the OCP codec does
    assert (got == ref).all()


def test_e4m3_encode_is_nearest_with_ties_to_even_by_brute_force():
    codes, vals = _finite_codes()
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(size=3000) * 30, rng.normal(size=3000) * 0.01])
    x = x.astype(np.float32)
    got = oracle.e4m3_from_f32(x)
    for xi, gi in zip(x.astype(np.float64), got):
        if abs(xi) >= 448:
            assert gi == (0xFE if xi < 0 else 0x7E)
            continue
        d = np.abs(vals - xi)
        best = d.min()
        cand = codes[d == best]
        # ties go to the even mantissa; among equal values (+0/-0) keep x's sign
        if len(cand) > 1:
            vals_c = oracle.e4m3_to_f64(cand)
            if (vals_c == 0).all():
                cand = cand[(cand >= 0x80) == (np.signbit(xi))]
            else:
                cand = cand[(cand & 1) == 0]
        assert len(cand) == 1 and gi == cand[0], (xi, gi, cand)


def test_e4m3_encode_midpoints_round_to_even():
    codes, vals = _finite_codes()
    pos = codes < 0x80
    c, v = codes[pos], vals[pos]
    order = np.argsort(v)
    c, v = c[order], v[order]
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)
    assert (mids.astype(np.float64) == (v[:-1] + v[1:]) / 2).all()  # exact in fp32
    got = oracle.e4m3_from_f32(mids)
    want = np.where((c[:-1] & 1) == 0, c[:-1], c[1:])
    assert (got == want).all()


def test_e4m3_encode_saturates_and_handles_nan():
    x = np.array([448.0, 449.0, 463.99, 464.0, 479.0, 480.0, 1e10, np.inf,
                  -449.0, -1e30, -np.inf, np.nan, -0.0, 0.0, 2.0 ** -10, 2.0 ** -10 * 1.0001],
                 np.float32)
    got = oracle.e4m3_from_f32(x)
    assert list(got[:8]) == [0x7E] * 8
    assert list(got[8:11]) == [0xFE] * 3
    assert got[11] == 0x7F
    assert got[12] == 0x80 and got[13] == 0x00
    assert got[14] == 0x00  # half of the smallest subnormal ties to zero (even)
    assert got[15] == 0x01


# -------------------------------------------------------------- layouts

def _build_paged(rng, lens, Hkv, D, bs, nb_extra=3, dtype=np.float16):
    """Contiguous per-sequence K/V and a scattered paged copy of them."""
    B = len(lens)
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + nb_extra
    MB = max(max(nblk), 1)
    perm = rng.permutation(NB)
    tables = np.full((B, MB), -1, np.int32)
    kc = np.full((NB, Hkv, bs, D), np.nan, dtype)
    vc = np.full((NB, Hkv, bs, D), np.nan, dtype)
    K, V = [], []
    cur = 0
    for b, L in enumerate(lens):
        tables[b, :nblk[b]] = perm[cur:cur + nblk[b]]
        cur += nblk[b]
        kb = rng.normal(size=(L, Hkv, D)).astype(dtype)
        vb = rng.normal(size=(L, Hkv, D)).astype(dtype)
        for p in range(L):
            kc[tables[b, p // bs], :, p % bs, :] = kb[p]
            vc[tables[b, p // bs], :, p % bs, :] = vb[p]
        K.append(kb)
        V.append(vb)
    return tables, kc, vc, K, V


def _dense(q, K, V, G, scale, start=0):
    """torch SDPA in fp64 on contiguous copies; GQA by repeating KV heads."""
    qd = torch.from_numpy(q.astype(np.float64))[:, None, :]           # Hq,1,D
    Kd = torch.from_numpy(K[start:].astype(np.float64)).permute(1, 0, 2)  # Hkv,L,D
    Vd = torch.from_numpy(V[start:].astype(np.float64)).permute(1, 0, 2)
    Kd = Kd.repeat_interleave(G, dim=0)
    Vd = Vd.repeat_interleave(G, dim=0)
    return F.scaled_dot_product_attention(qd, Kd, Vd, scale=scale)[:, 0].numpy()


def _odecode(q, kc, vc, tables, lens, Hkv, bs, scale, window=0, dt="f16", cdt=None, **kw):
    return oracle.decode(q.view(np.uint16), kc.view(np.uint16) if cdt != "fp8" else kc,
                         vc.view(np.uint16) if cdt != "fp8" else vc, tables,
                         np.asarray(lens, np.int32), num_kv_heads=Hkv, scale=scale,
                         block_size=bs, window=window, q_dtype=dt, cache_dtype=cdt or dt, **kw)


@pytest.mark.parametrize("G,D,bs", [(1, 32, 16), (4, 64, 16), (8, 32, 32), (2, 16, 8)])
def test_decode_matches_dense_sdpa(G, D, bs):
    rng = np.random.default_rng(100 + G + D + bs)
    Hkv = 2
    lens = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 97]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(len(lens), Hkv * G, D)).astype(np.float16)
    scale = D ** -0.5
    out = _odecode(q, kc, vc, tables, lens, Hkv, bs, scale)
    for b in range(len(lens)):
        ref = _dense(q[b], K[b], V[b], G, scale)
        assert np.abs(out[b] - ref).max() < 1e-13


def test_decode_window_matches_dense_on_the_last_w_positions():
    rng = np.random.default_rng(5)
    Hkv, G, D, bs = 2, 4, 32, 16
    lens = [1, 10, 40, 41, 100, 130]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(len(lens), Hkv * G, D)).astype(np.float16)
    for W in (1, 16, 40, 41, 1000):
        out = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.2, window=W)
        for b, L in enumerate(lens):
            start = max(0, L - W)
            ref = _dense(q[b], K[b], V[b], G, 0.2, start=start)
            assert np.abs(out[b] - ref).max() < 1e-13


def test_decode_window_equals_truncation():
    rng = np.random.default_rng(6)
    Hkv, G, D, bs = 1, 2, 16, 16
    lens = [50, 77]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(2, 2, D)).astype(np.float16)
    W = 20
    out_w = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.25, window=W)
    # fresh layout holding only the last W positions of each sequence
    rng2 = np.random.default_rng(60)
    short = [W, W]
    tables2, kc2, vc2, _, _ = _build_paged(rng2, short, Hkv, D, bs)
    for b, L in enumerate(lens):
        for i, p in enumerate(range(L - W, L)):
            kc2[tables2[b, i // bs], :, i % bs, :] = K[b][p]
            vc2[tables2[b, i // bs], :, i % bs, :] = V[b][p]
    out_t = _odecode(q, kc2, vc2, tables2, short, Hkv, bs, 0.25)
    assert np.array_equal(out_w, out_t)


def test_decode_invariant_under_block_id_permutation():
    rng = np.random.default_rng(8)
    Hkv, G, D, bs = 2, 2, 32, 16
    lens = [33, 64, 5]
    tables, kc, vc, _, _ = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(3, 4, D)).astype(np.float16)
    out1 = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.3)
    NB = kc.shape[0]
    sigma = rng.permutation(NB)  # block i moves to sigma[i]
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[sigma], vc2[sigma] = kc, vc
    tables2 = np.where(tables >= 0, sigma[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = _odecode(q, kc2, vc2, tables2, lens, Hkv, bs, 0.3)
    assert np.array_equal(out1, out2)


def test_decode_closed_forms():
    rng = np.random.default_rng(9)
    Hkv, G, D, bs = 1, 2, 8, 16
    # seq_len 1 returns V_0 exactly
    tables, kc, vc, K, V = _build_paged(rng, [1], Hkv, D, bs)
    q = rng.normal(size=(1, 2, D)).astype(np.float16)
    out = _odecode(q, kc, vc, tables, [1], Hkv, bs, 0.5)
    assert np.array_equal(out[0, 0], V[0][0, 0].astype(np.float64))
    assert np.array_equal(out[0, 1], V[0][0, 0].astype(np.float64))
    # identical K rows: uniform weights, output = mean of V
    L = 37
    tables, kc, vc, K, V = _build_paged(rng, [L], Hkv, D, bs)
    for p in range(L):
        kc[tables[0, p // bs], :, p % bs, :] = K[0][0]
    out = _odecode(q, kc, vc, tables, [L], Hkv, bs, 0.5)
    mean = V[0].astype(np.float64).mean(axis=0)[0]
    assert np.abs(out[0, 0] - mean).max() < 1e-14
    # q = 0: uniform weights
    tables, kc, vc, K, V = _build_paged(rng, [L], Hkv, D, bs)
    out = _odecode(np.zeros((1, 2, D), np.float16), kc, vc, tables, [L], Hkv, bs, 0.5)
    assert np.abs(out[0, 1] - V[0].astype(np.float64).mean(axis=0)[0]).max() < 1e-14
    # two positions with scores 2 and 0: weights 1/(1+e^-2) and 1/(1+e^2)
    tables, kc, vc, K, V = _build_paged(rng, [2], Hkv, D, bs)
    qq = np.zeros((1, 2, D), np.float16)
    qq[0, :, 0] = 1
    kc[tables[0, 0], 0, 0, :] = 0
    kc[tables[0, 0], 0, 0, 0] = 2
    kc[tables[0, 0], 0, 1, :] = 0
    out = _odecode(qq, kc, vc, tables, [2], Hkv, bs, 1.0)
    w0 = 1.0 / (1.0 + math.exp(-2.0))
    want = w0 * V[0][0, 0].astype(np.float64) + (1 - w0) * V[0][1, 0].astype(np.float64)
    assert np.abs(out[0, 0] - want).max() < 1e-14


def test_decode_empty_sequence_gives_zeros_and_gqa_groups_share_kv():
    rng = np.random.default_rng(10)
    Hkv, G, D, bs = 2, 4, 16, 16
    tables, kc, vc, K, V = _build_paged(rng, [0, 20], Hkv, D, bs)
    q = rng.normal(size=(2, 8, D)).astype(np.float16)
    q[1, 4:8] = q[1, 4]  # one KV group, identical queries
    out = _odecode(q, kc, vc, tables, [0, 20], Hkv, bs, 0.3)
    assert (out[0] == 0).all()
    assert all(np.array_equal(out[1, 4], out[1, h]) for h in range(5, 8))
    assert not np.array_equal(out[1, 0], out[1, 4])


def test_decode_bf16_and_fp8_match_dense_on_dequantised_values():
    rng = np.random.default_rng(12)
    Hkv, G, D, bs = 2, 4, 32, 16
    lens = [19, 64, 3]
    tables, kc16, vc16, K, V = _build_paged(rng, lens, Hkv, D, bs, dtype=np.float32)
    q = torch.from_numpy(rng.normal(size=(3, 8, D)).astype(np.float32)).to(torch.bfloat16)
    qbits = q.view(torch.int16).numpy().view(np.uint16)
    # bf16 cache
    kb = torch.from_numpy(kc16).to(torch.bfloat16)
    vb = torch.from_numpy(vc16).to(torch.bfloat16)
    out = oracle.decode(qbits, kb, vb, tables, np.array(lens, np.int32), num_kv_heads=Hkv,
                        scale=0.2, block_size=bs, q_dtype="bf16", cache_dtype="bf16")
    qd = q.double().numpy()
    for b, L in enumerate(lens):
        Kb = [torch.from_numpy(K[b]).to(torch.bfloat16).double().numpy()]
        Vb = [torch.from_numpy(V[b]).to(torch.bfloat16).double().numpy()]
        ref = _dense(qd[b], Kb[0], Vb[0], G, 0.2)
        assert np.abs(out[b] - ref).max() < 1e-13
    # e4m3 cache with per-tensor scales: value = decode(code) * scale
    ks, vs = 0.01, 0.02
    kcode = torch.from_numpy(np.nan_to_num(kc16 / ks)).to(torch.float8_e4m3fn).view(torch.uint8)
    vcode = torch.from_numpy(np.nan_to_num(vc16 / vs)).to(torch.float8_e4m3fn).view(torch.uint8)
    out8 = oracle.decode(qbits, kcode.numpy(), vcode.numpy(), tables, np.array(lens, np.int32),
                         num_kv_heads=Hkv, scale=0.2, block_size=bs, q_dtype="bf16",
                         cache_dtype="fp8", k_scale=ks, v_scale=vs)
    kdq = kcode.view(torch.float8_e4m3fn).double().numpy() * ks
    vdq = vcode.view(torch.float8_e4m3fn).double().numpy() * vs
    for b, L in enumerate(lens):
        Kd = np.stack([kdq[tables[b, p // bs], :, p % bs, :] for p in range(L)])
        Vd = np.stack([vdq[tables[b, p // bs], :, p % bs, :] for p in range(L)])
        ref = _dense(qd[b], Kd, Vd, G, 0.2)
        assert np.abs(out8[b] - ref).max() < 1e-13


def test_decode_pairs_subset_and_threads_agree():
    rng = np.random.default_rng(13)
    Hkv, G, D, bs = 2, 2, 16, 16
    lens = [40, 7, 90]
    tables, kc, vc, _, _ = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(3, 4, D)).astype(np.float16)
    full1 = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.3, threads=1)
    full4 = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.3, threads=4)
    assert np.array_equal(full1, full4)
    pairs = [(2, 3), (0, 1)]
    sub = _odecode(q, kc, vc, tables, lens, Hkv, bs, 0.3, pairs=pairs)
    for b, h in pairs:
        assert np.array_equal(sub[b, h], full1[b, h])


def test_decode_rejects_bad_block_id():
    rng = np.random.default_rng(14)
    tables, kc, vc, _, _ = _build_paged(rng, [20], 1, 8, 16)
    tables[0, 1] = kc.shape[0]
    with pytest.raises(ValueError):
        _odecode(np.zeros((1, 1, 8), np.float16), kc, vc, tables, [20], 1, 16, 1.0)


# ------------------------------------------------------------ write path

def test_reshape_16bit_scatter_skips_negative_slots_and_leaves_others():
    rng = np.random.default_rng(20)
    T, H, D, NB, bs = 7, 2, 8, 5, 4
    k = rng.normal(size=(T, H, D)).astype(np.float16)
    v = rng.normal(size=(T, H, D)).astype(np.float16)
    slots = np.array([3, -1, 17, 0, 19, -5, 8], np.int64)
    sentinel = np.uint16(0xABCD)
    kc = np.full((NB, H, bs, D), sentinel, np.uint16)
    vc = np.full((NB, H, bs, D), sentinel, np.uint16)
    oracle.reshape_and_cache(k, v, kc, vc, slots, "f16", "f16")
    touched = np.zeros((NB, bs), bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        touched[s // bs, s % bs] = True
        assert np.array_equal(kc[s // bs, :, s % bs, :], k[t].view(np.uint16))
        assert np.array_equal(vc[s // bs, :, s % bs, :], v[t].view(np.uint16))
    assert (kc.transpose(0, 2, 1, 3)[~touched] == sentinel).all()


def test_reshape_fp8_matches_torch_cast_of_fp32_quotient():
    rng = np.random.default_rng(21)
    T, H, D, NB, bs = 40, 2, 16, 4, 16
    k = torch.from_numpy(rng.normal(size=(T, H, D)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.normal(size=(T, H, D)).astype(np.float32) * 3).to(torch.bfloat16)
    ks, vs = 0.0123, 0.05
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    kc = np.full((NB, H, bs, D), 0x7F, np.uint8)
    vc = np.full((NB, H, bs, D), 0x7F, np.uint8)
    oracle.reshape_and_cache(k, v, kc, vc, slots, "bf16", "fp8", k_scale=ks, v_scale=vs)
    kq = (k.float() / torch.tensor(ks, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    vq = (v.float() / torch.tensor(vs, dtype=torch.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    for t, s in enumerate(slots):
        assert np.array_equal(kc[s // bs, :, s % bs, :], kq[t].numpy())
        assert np.array_equal(vc[s // bs, :, s % bs, :], vq[t].numpy())


# ------------------------------------------------- multi-token (causal)

def _odecode_multi(q, kc, vc, tables, lens, Hkv, bs, scale, window=0, dt="f16", **kw):
    return oracle.decode_multi(q.view(np.uint16), kc.view(np.uint16), vc.view(np.uint16), tables,
                               np.asarray(lens, np.int32), num_kv_heads=Hkv, scale=scale,
                               block_size=bs, window=window, q_dtype=dt, cache_dtype=dt, **kw)


@pytest.mark.parametrize("T,W", [(1, 0), (3, 0), (4, 0), (2, 0), (3, 20), (5, 7)])
def test_decode_multi_matches_dense_causal_sdpa(T, W):
    rng = np.random.default_rng(200 + T + W)
    Hkv, G, D, bs = 2, 2, 32, 16
    lens = [T, T + 1, 40, 17, 90]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(len(lens), T, Hkv * G, D)).astype(np.float16)
    out = _odecode_multi(q, kc, vc, tables, lens, Hkv, bs, 0.3, window=W)
    for b, L in enumerate(lens):
        # dense: queries at positions L-T..L-1, boolean causal (+ window) mask
        pos_q = np.arange(L - T, L)[:, None]
        pos_k = np.arange(L)[None, :]
        allowed = pos_k <= pos_q
        if W > 0:
            allowed &= pos_k > pos_q - W
        qd = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)       # Hq,T,D
        Kd = torch.from_numpy(K[b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        Vd = torch.from_numpy(V[b].astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = F.scaled_dot_product_attention(qd, Kd, Vd, attn_mask=torch.from_numpy(allowed),
                                             scale=0.3).permute(1, 0, 2).numpy()
        assert np.abs(out[b] - ref).max() < 1e-13


def test_decode_multi_rows_equal_single_query_decode_of_their_prefix():
    rng = np.random.default_rng(301)
    Hkv, G, D, bs, T = 2, 4, 16, 16, 3
    lens = [30, 3, 65]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q = rng.normal(size=(3, T, Hkv * G, D)).astype(np.float16)
    multi = _odecode_multi(q, kc, vc, tables, lens, Hkv, bs, 0.25, window=9)
    for t in range(T):
        single = _odecode(np.ascontiguousarray(q[:, t]), kc, vc, tables,
                          [L - T + t + 1 for L in lens], Hkv, bs, 0.25, window=9)
        assert np.array_equal(multi[:, t], single)


def test_decode_multi_queries_before_the_sequence_give_zeros():
    rng = np.random.default_rng(302)
    tables, kc, vc, K, V = _build_paged(rng, [2], 1, 8, 16)
    q = rng.normal(size=(1, 4, 1, 8)).astype(np.float16)
    out = _odecode_multi(q, kc, vc, tables, [2], 1, 16, 1.0)
    assert (out[0, :2] == 0).all() and (out[0, 2:] != 0).any()


def test_repeated_rows_in_a_request_are_computed_once_and_correctly():
    """Requests that list a row twice (random samples do) give the same
    values as requests that list it once: the rows are computed on parallel
    threads, which must never share an output row."""
    rng = np.random.default_rng(303)
    Hkv, G, D, bs, T = 2, 2, 16, 16, 3
    lens = [70, 33]
    tables, kc, vc, K, V = _build_paged(rng, lens, Hkv, D, bs)
    q3 = rng.normal(size=(2, Hkv * G, D)).astype(np.float16)
    pairs = [(1, 3)] * 64 + [(0, 0)] * 64
    once = _odecode(q3, kc, vc, tables, lens, Hkv, bs, 0.2, pairs=[(1, 3), (0, 0)])
    many = _odecode(q3, kc, vc, tables, lens, Hkv, bs, 0.2, pairs=pairs)
    assert np.array_equal(once, many)
    q4 = rng.normal(size=(2, T, Hkv * G, D)).astype(np.float16)
    tr = [(1, 2, 3)] * 64 + [(0, 1, 0)] * 64
    once = _odecode_multi(q4, kc, vc, tables, lens, Hkv, bs, 0.2,
                          triples=[(1, 2, 3), (0, 1, 0)])
    many = _odecode_multi(q4, kc, vc, tables, lens, Hkv, bs, 0.2, triples=tr)
    assert np.array_equal(once, many)
