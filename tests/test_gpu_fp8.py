"""GPU: FP8 (E4M3) K/V pages with per-channel scales.

Writes are integer work: every stored code must equal the FP8 oracle's
quantisation (oracle/fp8.py) of the row written at that slot, bit for bit.
Decode over FP8 pages is compared with the attention oracle run over the
oracle's dequantised K/V (code * scale, float64) at the usual bf16 bar."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import fp8, transfer
from _gpu_common import compare, f64, gpu_ready, ncores, pol_tuple, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL
D = 128


def _mk(hq, hkv, P, seqs, max_len, pages, layers=1, kv_dtype=1, d=D, max_idx=8192):
    from head_aware_paged_gb300 import Config, SegPagedCache
    return SegPagedCache(Config(num_layers=layers, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                                page_size=P, max_seqs=seqs, max_seq_len=max_len, num_pages=pages,
                                max_idx_per_seq=max_idx, max_tokens=max_len, max_batch=seqs,
                                kv_dtype=kv_dtype))


def _outlier_kv(n, hkv, seed):
    """K with a few outlier channels per head (the case per-channel scales
    are for), V plain normal; bf16 on the device."""
    k = W.normal((n, hkv, D), W.tensor_seed(seed, "k"), 0.5, device="cuda")
    v = W.normal((n, hkv, D), W.tensor_seed(seed, "v"), device="cuda")
    boost = torch.ones(hkv, D, device="cuda")
    for h in range(hkv):                 # the same outlier channels for every call
        boost[h, np.random.default_rng(1234 + h).choice(D, 4, replace=False)] = 12.0
    return (k.float() * boost).to(torch.bfloat16), v


def _scales(x):
    """Per (head, channel) absmax / 448 over x [n, hkv, d], inside the
    accepted range [2^-14, 128]."""
    a = x.float().abs().amax(dim=0).cpu().numpy().astype(np.float64)
    return np.clip(a / 448.0, 2.0 ** -14, 128.0).astype(np.float32)


def _stored(cache, seq, layer, h):
    ids, pos = cache.export_table(seq, layer, h)
    rows = [(p, pg, s) for pg, slots in zip(ids, pos) for s, p in enumerate(slots) if p >= 0]
    return rows


def _check_codes(cache, seq, layer, h, k, v, ks, vs):
    rows = _stored(cache, seq, layer, h)
    if not rows:
        return 0
    pos = np.array([r[0] for r in rows])
    pg = torch.tensor([r[1] for r in rows], device="cuda")
    sl = torch.tensor([r[2] for r in rows], device="cuda")
    got_k = cache.k_pool()[pg, sl].cpu().numpy()
    got_v = cache.v_pool()[pg, sl].cpu().numpy()
    want_k = fp8.quantize(f64(k[:, h])[pos], ks[h])
    want_v = fp8.quantize(f64(v[:, h])[pos], vs[h])
    np.testing.assert_array_equal(got_k, want_k)
    np.testing.assert_array_equal(got_v, want_v)
    return len(rows)


def _dq(x, s):
    """Oracle dequantisation of dense rows x [n, hkv, d] with scales [hkv, d]."""
    xs = f64(x)
    out = np.empty_like(xs)
    for h in range(xs.shape[1]):
        out[:, h] = fp8.dequantize(fp8.quantize(xs[:, h], s[h]), s[h])
    return out


@pytest.mark.parametrize("P,hq,hkv", [(64, 32, 8), (16, 8, 2), (128, 16, 2), (32, 24, 8)])
def test_codes_bit_exact_and_decode_parity(P, hq, hkv):
    gpu_ready()
    rng = np.random.default_rng(P + hq)
    B, max_len = 4, 3000
    lens = [int(x) for x in rng.integers(1, max_len, size=B)]
    lens[0], lens[1] = 1, max_len - 1
    cache = _mk(hq, hkv, P, B, max_len, B * hkv * (max_len // P + 2))
    data, pols = [_outlier_kv(lens[b], hkv, 100 + b) for b in range(B)], []
    ks = _scales(torch.cat([k for k, _ in data]))
    vs = _scales(torch.cat([v for _, v in data]))
    cache.set_kv_scales(0, ks, vs)
    for b in range(B):
        row = []
        for h in range(hkv):
            kind = int(rng.integers(0, 3))
            if kind == G:
                row.append(W.HeadPolicy(G))
            elif kind == L:
                row.append(W.HeadPolicy(L, int(rng.integers(0, 9)), int(rng.integers(1, 700))))
            else:
                idx = np.sort(rng.choice(max_len, int(rng.integers(0, 400)), replace=False))
                row.append(W.HeadPolicy(R, idx=idx.astype(np.int32)))
        pols.append(row)
        cache.set_policy(b, to_c_policies([row]))
        cache.build(b, 0, *data[b])
    torch.cuda.synchronize()
    assert cache.status() == 0
    checked = sum(_check_codes(cache, b, 0, h, *data[b], ks, vs) for b in range(B) for h in range(hkv))
    assert checked > 0
    q = W.normal((B, hq, D), 99, device="cuda")
    out, lse = cache.decode(0, list(range(B)), q)
    for b in range(B):
        pt = [pol_tuple(p) for p in pols[b]]
        ref, lref = oracle.attend(f64(q[b:b + 1]), _dq(data[b][0], ks), _dq(data[b][1], vs),
                                  [lens[b] - 1], pt, "f64", threads=ncores())
        compare(out[b:b + 1], ref, lse[b:b + 1], lref, "fp8 seq %d" % b)
    assert cache.status() == 0


def test_append_steps_long_context():
    """Build 20K tokens, then append-one + decode steps; codes of the
    appended rows and the decode (many splits per unit) against the oracle."""
    gpu_ready()
    hq, hkv, P, n0, steps = 32, 8, 64, 20000, 3
    cache = _mk(hq, hkv, P, 1, n0 + 64, hkv * ((n0 + 64) // P + 2))
    pols = [W.HeadPolicy(G), W.HeadPolicy(L, 4, 1024), W.HeadPolicy(G), W.HeadPolicy(G),
            W.HeadPolicy(R, idx=np.arange(0, n0 + steps, 7, dtype=np.int32)), W.HeadPolicy(G),
            W.HeadPolicy(L, 0, 333), W.HeadPolicy(G)]
    cache.set_policy(0, to_c_policies([pols]))
    k, v = _outlier_kv(n0 + steps, hkv, 77)
    ks, vs = _scales(k), _scales(v)
    cache.set_kv_scales(0, ks, vs)
    cache.build(0, 0, k[:n0].contiguous(), v[:n0].contiguous())
    pt = [pol_tuple(p) for p in pols]
    kd, vd = _dq(k, ks), _dq(v, vs)
    for s in range(steps):
        t = n0 + s
        cache.append_kv(0, [0], [0, 1], k[t:t + 1].contiguous(), v[t:t + 1].contiguous())
        q = W.normal((1, hq, D), 500 + s, device="cuda")
        out, lse = cache.decode(0, [0], q)
        ref, lref = oracle.attend(f64(q), kd[:t + 1], vd[:t + 1], [t], pt, "f64", threads=ncores())
        compare(out, ref, lse, lref, "fp8 step %d" % s)
    torch.cuda.synchronize()
    for h in range(hkv):
        _check_codes(cache, 0, 0, h, k[:n0 + steps], v[:n0 + steps], ks, vs)
    assert cache.status() == 0


@pytest.mark.parametrize("P,n,c2", [(64, 700, 300), (16, 1500, 200), (128, 5000, 129), (32, 33, 640)])
def test_prefill_first_chunk_then_over_fp8_history(P, n, c2):
    """A first chunk prefills over its own bf16 K/V and its write stores
    codes; the next chunk attends over the FP8 history (dequantised by the
    oracle) plus its own bf16 rows."""
    gpu_ready()
    hq, hkv = 16, 4
    tot = n + c2
    cache = _mk(hq, hkv, P, 2, 2 * tot + 64, 2 * hkv * ((tot + 64) // P + 3))   # max_tokens >= both chunks
    pols = [W.HeadPolicy(G), W.HeadPolicy(L, 4, 100), W.HeadPolicy(G),
            W.HeadPolicy(R, idx=np.arange(3, tot, 5, dtype=np.int32))]
    cache.set_policy(0, to_c_policies([pols]))
    cache.set_policy(1, to_c_policies([pols]))
    q = W.normal((2 * tot, hq, D), 1 + P, device="cuda")
    k, v = _outlier_kv(2 * tot, hkv, 2 + P)
    ks, vs = _scales(k), _scales(v)
    cache.set_kv_scales(0, ks, vs)
    pt = [pol_tuple(p) for p in pols]
    # first chunk: rows 0..n-1 of both sequences (sequence b uses rows b*tot ..)
    r1 = torch.cat([torch.arange(b * tot, b * tot + n) for b in range(2)]).cuda()
    q1, k1, v1 = q[r1].contiguous(), k[r1].contiguous(), v[r1].contiguous()
    out, lse = cache.prefill(0, [0, 1], [0, n, 2 * n], q1, k1, v1)
    torch.cuda.synchronize()
    for b in range(2):
        sl = slice(b * n, (b + 1) * n)
        ref, lref = oracle.attend(f64(q1[sl]), f64(k1[sl]), f64(v1[sl]), list(range(n)), pt, "f64",
                                  threads=ncores())
        compare(out[sl], ref, lse[sl], lref, "fp8 first chunk %d" % b)
    cache.append_kv(0, [0, 1], [0, n, 2 * n], k1, v1)
    torch.cuda.synchronize()
    for b in range(2):
        sl = slice(b * n, (b + 1) * n)
        assert sum(_check_codes(cache, b, 0, h, k1[sl], v1[sl], ks, vs) for h in range(hkv)) > 0
    # second chunk over the FP8 history
    r2 = torch.cat([torch.arange(b * tot + n, (b + 1) * tot) for b in range(2)]).cuda()
    q2, k2, v2 = q[r2].contiguous(), k[r2].contiguous(), v[r2].contiguous()
    out2, lse2 = cache.prefill(0, [0, 1], [0, c2, 2 * c2], q2, k2, v2)
    torch.cuda.synchronize()
    for b in range(2):
        hist = slice(b * tot, b * tot + n)
        kk = np.concatenate([_dq(k[hist], ks), f64(k2[b * c2:(b + 1) * c2])], axis=0)
        vv = np.concatenate([_dq(v[hist], vs), f64(v2[b * c2:(b + 1) * c2])], axis=0)
        sl = slice(b * c2, (b + 1) * c2)
        ref, lref = oracle.attend(f64(q2[sl]), kk, vv, list(range(n, tot)), pt, "f64", threads=ncores())
        compare(out2[sl], ref, None, None, "fp8 history chunk %d" % b)
        # The history rows enter the bf16 MMAs as bf16(code * scale): each
        # score moves by at most 2^-9 sum_i |q_i k_i| / sqrt(d) (twice that
        # as slack), and so does the log-sum-exp
        qa = np.abs(f64(q2[sl]))                              # [c2, hq, d]
        ka = np.abs(kk[:n])                                   # [n, hkv, d]
        grp = hq // hkv
        bound = np.stack([(qa[:, h] @ ka[:, h // grp].T).max(axis=1) for h in range(hq)], axis=1)
        bound = 2.0 ** -8 * bound / np.sqrt(D) + 2e-3
        lg = lse2[sl].cpu().numpy().astype(np.float64)
        fin = np.isfinite(lref)
        assert np.array_equal(np.isfinite(lg), fin)
        assert (np.abs(lg - lref)[fin] <= bound[fin]).all(), np.abs(lg - lref)[fin].max()
    assert cache.status() == 0


def test_pack_unpack_round_trip():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    hq, hkv, P, n = 8, 2, 32, 900
    a = _mk(hq, hkv, P, 2, 1024, 200)
    pols = [W.HeadPolicy(L, 3, 200), W.HeadPolicy(R, idx=np.array([1, 5, 99, 500, 899], np.int32))]
    a.set_policy(1, to_c_policies([pols]))
    k, v = _outlier_kv(n, hkv, 3)
    ks, vs = _scales(k), _scales(v)
    a.set_kv_scales(0, ks, vs)
    a.build(1, 0, k, v)
    buf = a.pack(1)
    torch.cuda.synchronize()
    h = buf[:96].cpu().numpy().view(np.int64)
    assert h[11] == 1                                   # kv_dtype
    pt = [[pol_tuple(p) for p in pols]]
    codes_k = np.stack([fp8.quantize(f64(k[:, i]), ks[i]) for i in range(hkv)], axis=1)
    codes_v = np.stack([fp8.quantize(f64(v[:, i]), vs[i]) for i in range(hkv)], axis=1)
    want = transfer.payload(pt, [n], [codes_k], [codes_v], P)
    got = buf[int(h[8]):int(h[10])].cpu().numpy()
    np.testing.assert_array_equal(got, want)
    b = _mk(hq, hkv, P, 3, 1024, 300)
    b.set_kv_scales(0, ks, vs)
    b.unpack(2, buf)
    q = W.normal((1, hq, D), 4, device="cuda")
    oa, la = a.decode(0, [1], q)
    ob, lb = b.decode(0, [2], q)
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    # a bf16 receiver refuses an FP8 buffer
    with pytest.raises(SegPagedError):
        _mk(hq, hkv, P, 2, 1024, 200, kv_dtype=0).unpack(0, buf)
    assert a.status() == 0 and b.status() == 0


def test_scale_and_config_validation():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError
    hkv = 2
    c = _mk(4, hkv, 16, 1, 256, 64)
    ok = np.full((hkv, D), 0.01, np.float32)
    for bad in (0.0, -1.0, np.nan, np.inf, 200.0, 2.0 ** -15):
        s = ok.copy()
        s[1, 7] = bad
        with pytest.raises(SegPagedError):
            c.set_kv_scales(0, s, ok)
        with pytest.raises(SegPagedError):
            c.set_kv_scales(0, ok, s)
    c.set_kv_scales(0, ok, ok)
    c.set_kv_scales(0, np.full((hkv, D), 128.0, np.float32), np.full((hkv, D), 2.0 ** -14, np.float32))
    c.set_policy(0, to_c_policies([[W.HeadPolicy(G)] * hkv]))
    c.build(0, 0, *(W.normal((10, hkv, D), s, device="cuda") for s in (1, 2)))
    with pytest.raises(SegPagedError):      # pages already hold codes under the old scales
        c.set_kv_scales(0, ok, ok)
    with pytest.raises(SegPagedError):      # scales belong to FP8 caches only
        _mk(4, hkv, 16, 1, 256, 64, kv_dtype=0).set_kv_scales(0, ok, ok)
    for kw in ({"d": 64}, {"kv_dtype": 2}):
        with pytest.raises(SegPagedError):
            _mk(4, hkv, 16, 1, 256, 64, **kw)
    assert c.status() == 0


@pytest.mark.parametrize("P", [64, 16])
def test_rope_realign_of_fp8_pages_matches_the_oracle_bit_for_bit(P):
    """RoPE realignment of FP8 keys: every rotated code equals the oracle's
    (dequantise with the channel scales, rotate in float32 without fused
    operations, quantise like a write); rows outside the position range,
    other sequences, other layers and V are untouched."""
    gpu_ready()
    from oracle import rope
    hq, hkv, n = 8, 4, 700
    cache = _mk(hq, hkv, P, 2, n + 64, 2 * 2 * hkv * (n // P + 4), layers=2)
    pols = [W.HeadPolicy(G), W.HeadPolicy(L, 5, 70), W.HeadPolicy(G),
            W.HeadPolicy(R, idx=np.array(sorted({3, 40, 41, 99, 250, 251, 400, 699}), np.int32))]
    data = {}
    for sq in range(2):
        cache.set_policy(sq, to_c_policies([pols, pols]))
    for l in range(2):
        k, v = _outlier_kv(2 * n, hkv, 40 + l)
        ks, vs = _scales(k), _scales(v)
        cache.set_kv_scales(l, ks, vs)
        data[l] = (ks, vs)
        for sq in range(2):
            cache.build(sq, l, k[sq * n:(sq + 1) * n].contiguous(), v[sq * n:(sq + 1) * n].contiguous())
    torch.cuda.synchronize()
    k0 = cache.k_pool().clone()
    v0 = cache.v_pool().clone()
    lo, hi, delta = 30, 650, 98765
    cache.rope_realign(1, [0], delta, pos_lo=lo, pos_hi=hi)
    torch.cuda.synchronize()
    assert cache.status() == 0
    assert torch.equal(cache.v_pool(), v0)
    k1 = cache.k_pool()
    touched = torch.zeros(k1.shape[:2], dtype=torch.bool, device="cuda")
    ks = data[1][0]
    for h in range(hkv):
        sel = [(p, pg, sl) for p, pg, sl in _stored(cache, 0, 1, h) if lo <= p < hi]
        assert sel
        pg = torch.tensor([r[1] for r in sel], device="cuda")
        sl = torch.tensor([r[2] for r in sel], device="cuda")
        want = rope.realign_fp8(k0[pg, sl].cpu().numpy(), ks[h], delta)
        np.testing.assert_array_equal(k1[pg, sl].cpu().numpy(), want)
        touched[pg, sl] = True
    assert torch.equal(k1[~touched], k0[~touched])
