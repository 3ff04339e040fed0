"""GPU: pack / unpack of a sequence's trimmed pages (sp_pack_seq /
sp_unpack_seq) against the transfer oracle (oracle/transfer.py)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import transfer
from _gpu_common import gpu_ready, to_c_policies

pytestmark = pytest.mark.gpu

G, L, R = W.GLOBAL, W.LOCAL, W.RETRIEVAL
MAGIC = 0x3156504B50535053


def _cache(d=64, P=16, pages=200, seqs=2, max_len=512, layers=2, hkv=3):
    from head_aware_paged_gb300 import Config, SegPagedCache
    return SegPagedCache(Config(num_layers=layers, num_q_heads=2 * hkv, num_kv_heads=hkv, head_dim=d,
                                page_size=P, max_seqs=seqs, max_seq_len=max_len, num_pages=pages,
                                max_idx_per_seq=1024, max_tokens=max_len, max_batch=seqs))


def _policies():
    idx = np.array([2, 9, 10, 64, 100, 101, 250, 300, 333], np.int32)
    return [[W.HeadPolicy(G), W.HeadPolicy(L, 4, 40), W.HeadPolicy(R, idx=idx)],
            [W.HeadPolicy(L, 20, 33), W.HeadPolicy(G), W.HeadPolicy(R, idx=idx[::2].copy())]]


def _fill(cache, seq, pols, d, seed):
    """Layer 0: built from 300 dense rows; layer 1: 300 rows then 37 appended
    (the LOCAL ring wraps).  Returns the dense K/V of every layer."""
    cache.set_policy(seq, to_c_policies(pols))
    ks, vs = [], []
    for l, n0, extra in ((0, 300, 0), (1, 300, 37)):
        k = W.normal((n0 + extra, 3, d), W.tensor_seed(seed, "k", l), device="cuda")
        v = W.normal((n0 + extra, 3, d), W.tensor_seed(seed, "v", l), device="cuda")
        cache.build(seq, l, k[:n0].contiguous(), v[:n0].contiguous())
        if extra:
            cache.append_kv(l, [seq], [0, extra], k[n0:].contiguous(), v[n0:].contiguous())
        ks.append(k)
        vs.append(v)
    torch.cuda.synchronize()
    return ks, vs


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy()


def _header(buf):
    h = buf[:96].cpu().numpy().view(np.int64)
    return dict(zip(["magic", "version", "layers", "hkv", "head_dim", "page_size", "n_units",
                     "idx_total", "payload_off", "payload_bytes", "total_bytes", "kv_dtype"], h.tolist()))


def test_pack_matches_oracle_bit_exact():
    gpu_ready()
    d, P = 64, 16
    cache = _cache(d, P)
    pols = _policies()
    ks, vs = _fill(cache, 1, pols, d, 5)
    buf = cache.pack(1)
    torch.cuda.synchronize()
    assert cache.status() == 0
    h = _header(buf)
    assert h["magic"] == MAGIC and h["version"] == 1
    assert (h["layers"], h["hkv"], h["head_dim"], h["page_size"], h["n_units"]) == (2, 3, d, P, 6)
    assert h["total_bytes"] == buf.numel() and h["payload_off"] % 256 == 0
    assert h["kv_dtype"] == 0
    n_layer = buf[96:96 + 16].cpu().numpy().view(np.int64).tolist()
    assert n_layer == [300, 337]
    pt = [[(p.kind, p.sink, p.window, None if p.idx is None else p.idx.tolist()) for p in row]
          for row in pols]
    want = transfer.payload(pt, n_layer, [_bits(k) for k in ks], [_bits(v) for v in vs], P)
    got = buf[h["payload_off"]:h["total_bytes"]].cpu().numpy().view(np.int16)
    assert got.size == want.size
    np.testing.assert_array_equal(got, want)
    # size query equals the real size; dense / packed ratio as the oracle counts it
    from head_aware_paged_gb300 import sp_pack_seq
    assert sp_pack_seq(cache.handle, 1, None) == buf.numel()
    assert h["payload_bytes"] * transfer.transfer_ratio(pt, n_layer, P) == pytest.approx(
        sum(n_layer) * 3 * 2 * d * 2)


def test_unpack_round_trip_equal_state_and_attention():
    gpu_ready()
    d, P = 64, 16
    a = _cache(d, P)
    pols = _policies()
    ks, vs = _fill(a, 0, pols, d, 9)
    buf = a.pack(0)
    b = _cache(d, P, pages=300, seqs=3)
    # occupy some pages first so the receiver's page ids differ from the sender's
    b.set_policy(0, to_c_policies([[W.HeadPolicy(G)] * 3] * 2))
    b.build(0, 0, *(W.normal((40, 3, d), s, device="cuda") for s in (1, 2)))
    b.unpack(2, buf)
    torch.cuda.synchronize()
    assert b.status() == 0
    for l in range(2):
        assert b.seq_len(2, l) == a.seq_len(0, l)
        for h in range(3):
            ia, pa = a.export_table(0, l, h)
            ib, pb = b.export_table(2, l, h)
            assert pa == pb, (l, h)
            assert len(ia) == len(ib)
    # the next decode token and a prefill chunk give bitwise the same results
    q = W.normal((1, 6, d), 31, device="cuda")
    kn = W.normal((1, 3, d), 32, device="cuda")
    vn = W.normal((1, 3, d), 33, device="cuda")
    for l in range(2):
        a.append_kv(l, [0], [0, 1], kn, vn)
        b.append_kv(l, [2], [0, 1], kn, vn)
        oa, la = a.decode(l, [0], q)
        ob, lb = b.decode(l, [2], q)
        assert torch.equal(oa, ob) and torch.equal(la, lb)
    qc = W.normal((20, 6, d), 34, device="cuda")
    kc = W.normal((20, 3, d), 35, device="cuda")
    vc = W.normal((20, 3, d), 36, device="cuda")
    oa, la = a.prefill(1, [0], [0, 20], qc, kc, vc)
    ob, lb = b.prefill(1, [2], [0, 20], qc, kc, vc)
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    assert a.status() == 0 and b.status() == 0


def test_refusals_change_nothing():
    gpu_ready()
    from head_aware_paged_gb300 import SegPagedError, sp_pack_seq
    d, P = 64, 16
    a = _cache(d, P)
    _fill(a, 0, _policies(), d, 3)
    buf = a.pack(0)
    # too small a destination
    small = torch.empty(256 * 1024, dtype=torch.uint8, device="cuda")[:1024]
    with pytest.raises(SegPagedError):
        sp_pack_seq(a.handle, 0, small)
    # another head_dim or page size
    for kw in ({"d": 128}, {"P": 32}):
        with pytest.raises(SegPagedError):
            _cache(**kw).unpack(0, buf)
    # an occupied slot
    b = _cache(d, P)
    b.set_policy(0, to_c_policies([[W.HeadPolicy(G)] * 3] * 2))
    b.build(0, 0, *(W.normal((10, 3, d), s, device="cuda") for s in (1, 2)))
    with pytest.raises(SegPagedError):
        b.unpack(0, buf)
    # not enough pages: nothing changes
    c = _cache(d, P, pages=20)
    free0 = c.free_pages()
    with pytest.raises(SegPagedError, match="pages"):
        c.unpack(1, buf)
    assert c.free_pages() == free0 and c.seq_len(1, 0) == 0 and c.seq_len(1, 1) == 0
    # a corrupted header
    bad = buf.clone()
    bad[0] ^= 1
    with pytest.raises(SegPagedError):
        _cache(d, P).unpack(0, bad)
    assert a.status() == 0
