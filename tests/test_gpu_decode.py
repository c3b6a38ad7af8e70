"""flat_decode_attn against the oracle on hand-built flat caches.

The caches are built directly (no scoring or compaction) so that the per-head lengths can
be pushed to the cases the decode kernels have to get right: empty heads, one-row heads, heads
longer than a whole row chunk (their partials are merged across CTAs), heads sharing a
chunk, reserve rows exhausted, and every lane layout (16-byte slices per row of 1, 2, 4, 8,
16 and 32) and group size 1, 2, 3, 4, 8.  Every case runs through each decode kernel that
takes its shape (256-byte rows for all but the row-balanced split; the other shapes fall
through to it).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O

from .kvpath import assert_decode_close, np64, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["split", "heads", "rows", "parts"], autouse=True)
def decode_path(request):
    """Every case through the four decode kernels: the one-launch split of the used rows
    across CTAs (256-byte rows, G <= 4, short heads), one CTA per KV head (256-byte rows, the
    other groups), the row-balanced split (the rest) and the heads in parts (256-byte rows,
    G <= 4, at most 512 heads).  A shape a forced kernel does not take goes to the
    one-CTA-per-head kernel, else the row-balanced split."""
    old = os.environ.get("KVEVICT_DECODE_PATH")
    os.environ["KVEVICT_DECODE_PATH"] = request.param
    yield request.param
    if old is None:
        os.environ.pop("KVEVICT_DECODE_PATH", None)
    else:
        os.environ["KVEVICT_DECODE_PATH"] = old


def build_cache(B, L, hkv, G, d, lens, reserve, dtype, seed):
    """Flat cache with the given per-head lengths; rows past lens hold junk (never read)."""
    gen = torch.Generator().manual_seed(seed)
    H = B * L * hkv
    lens = np.asarray(lens, dtype=np.int64)
    assert lens.shape == (H,)
    ext = lens + reserve
    flat = np.concatenate([[0], np.cumsum(ext)])
    cu = np.stack([flat[s * hkv: s * hkv + hkv + 1] for s in range(B * L)])
    cap = int(flat[-1])
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    kf = torch.randn(cap, d, generator=gen).to(tdt)
    vf = (torch.randn(cap, d, generator=gen) * torch.exp(0.5 * torch.randn(cap, 1, generator=gen))).to(tdt)
    tau = torch.exp(torch.rand(B, L, hkv * G, 1, generator=gen) * math.log(8.0)) * 0.5
    q = (torch.randn(B, L, hkv * G, d, generator=gen) * tau).to(tdt)
    kn = torch.randn(B, L, hkv, d, generator=gen).to(tdt)
    vn = torch.randn(B, L, hkv, d, generator=gen).to(tdt)
    return dict(kf=kf, vf=vf, q=q, kn=kn, vn=vn, cu=torch.from_numpy(cu.copy()),
                lens=torch.from_numpy(lens.astype(np.int32)), cap=cap)


def oracle_decode(c, B, L, hkv, scale, append):
    Kf, Vf = np64(c["kf"]), np64(c["vf"])
    lens = c["lens"].numpy().astype(np.int64).reshape(B, L, hkv)
    cu = c["cu"].numpy().reshape(B, L, hkv + 1)
    outs = np.zeros(tuple(c["q"].shape))
    new_lens = lens.copy()
    for b in range(B):
        for l in range(L):
            kn = np64(c["kn"][b, l]) if append else None
            vn = np64(c["vn"][b, l]) if append else None
            o, Kf2, Vf2, ln = _flat_decode_partial(np64(c["q"][b, l]), Kf, Vf, cu[b, l], lens[b, l],
                                                   scale, kn, vn)
            outs[b, l] = o
            new_lens[b, l] = ln
            Kf, Vf = Kf2, Vf2
    return outs, new_lens


def _flat_decode_partial(q, Kf, Vf, cu, lens, scale, kn, vn):
    """The oracle's decode step, with the append skipped for heads that have no reserve row."""
    if kn is None:
        return O.flat_decode(q, Kf, Vf, cu, lens, scale)
    hkv = len(lens)
    ok = cu[:-1] + lens < cu[1:]
    Kf = Kf.copy()
    Vf = Vf.copy()
    lens = lens.copy()
    for g in range(hkv):
        if ok[g]:
            Kf[cu[g] + lens[g]] = kn[g]
            Vf[cu[g] + lens[g]] = vn[g]
            lens[g] += 1
    o, _, _, _ = O.flat_decode(q, Kf, Vf, cu, lens, scale)
    return o, Kf, Vf, lens


def check(c, B, L, hkv, G, d, dtype, append, expect_code=0):
    dev = "cuda"
    shape = kv.KvShape.of(batch=B, layers=L, hq=hkv * G, hkv=hkv, d=d, n=100000, w=1, pool=1,
                          dtype=dtype)
    scale = 1.0 / math.sqrt(d)
    ref, ref_lens = oracle_decode(c, B, L, hkv, scale, append)
    kf, vf = c["kf"].to(dev), c["vf"].to(dev)
    cu, lens = c["cu"].to(dev), c["lens"].to(dev)
    q = c["q"].to(dev)
    out = torch.full_like(q, float("nan"))
    ws = workspace(kv.KV_OP_DECODE, shape)
    kn = c["kn"].to(dev) if append else None
    vn = c["vn"].to(dev) if append else None
    kv.flat_decode_attn(shape, q, kn, vn, kf, vf, cu, lens, scale, out, ws)
    code = kv.kv_check_device_status(ws)
    assert code == expect_code
    got = np64(out)
    assert np.isfinite(got).all()
    assert_decode_close(got, ref, dtype)
    np.testing.assert_array_equal(lens.cpu().numpy().reshape(B, L, hkv), ref_lens)
    if append:
        # the appended rows are exact copies of k_new / v_new
        cu_h = c["cu"].numpy()
        l0 = c["lens"].numpy().reshape(B, L, hkv)
        for b in range(B):
            for l in range(L):
                for g in range(hkv):
                    r = cu_h[b * L + l, g] + l0[b, l, g]
                    if r < cu_h[b * L + l, g + 1]:
                        assert torch.equal(kf[r].cpu(), c["kn"][b, l, g])
                        assert torch.equal(vf[r].cpu(), c["vn"][b, l, g])


CASES = [
    # (dtype, d, G, hkv) -- slices per row: bf16 d/8, f32 d/4
    ("bf16", 128, 4, 4),    # 16 slices, transposed reduction, G = 4
    ("bf16", 128, 8, 2),    # 16 slices, transposed reduction, G = 8
    ("f32", 64, 4, 2),      # 16 slices, fp32
    ("bf16", 64, 3, 2),     # 8 slices, butterfly reduction, G = 3 padded to 4
    ("f32", 32, 1, 4),      # 8 slices, G = 1
    ("bf16", 8, 2, 3),      # 1 slice per row
    ("f32", 128, 2, 2),     # 32 slices per row
    ("bf16", 96, 4, 2),     # 12 slices: lanes 12..15 of each row idle
    # 256-byte rows with small groups: tiles of 16 rows (G padded to 2) and a padded G = 3
    ("bf16", 128, 1, 8),
    ("bf16", 128, 2, 4),
    ("f32", 64, 2, 2),
    ("bf16", 128, 3, 2),
]


@pytest.mark.parametrize("dtype,d,G,hkv", CASES)
@pytest.mark.parametrize("append", [True, False])
def test_decode_uneven_heads(dtype, d, G, hkv, append):
    B, L = 2, 2
    H = B * L * hkv
    rng = np.random.default_rng(d * 31 + G * 7 + hkv + int(append))
    # heads of 0 and 1 rows, short heads, and heads longer than any row chunk
    base = [0, 1, 3, 5000, 17, 1200, 64, 2]
    lens = np.array([base[i % len(base)] for i in range(H)], dtype=np.int64)
    lens = np.where(rng.random(H) < 0.3, rng.integers(0, 300, H), lens)
    c = build_cache(B, L, hkv, G, d, lens, reserve=3, dtype=dtype, seed=int(rng.integers(1 << 30)))
    check(c, B, L, hkv, G, d, dtype, append)


def test_decode_no_reserve_left():
    """Heads with no reserve row skip the append (device check 3) and attend without it."""
    B, L, hkv, G, d = 1, 2, 4, 4, 128
    lens = np.array([10, 700, 0, 33, 5, 6, 7, 4000])
    c = build_cache(B, L, hkv, G, d, lens, reserve=0, dtype="bf16", seed=5)
    check(c, B, L, hkv, G, d, "bf16", append=True, expect_code=3)


def test_decode_many_small_heads_per_chunk():
    """Hundreds of tiny heads: one CTA walks more than one table of heads."""
    B, L, hkv, G, d = 1, 40, 8, 4, 128
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 2, B * L * hkv)
    c = build_cache(B, L, hkv, G, d, lens, reserve=1, dtype="bf16", seed=6)
    check(c, B, L, hkv, G, d, "bf16", append=True)


@pytest.mark.parametrize("lens", [[0, 1, 2, 5], [0, 0, 0, 0], [40, 0, 1, 0]])
def test_decode_fewer_rows_than_ctas(lens):
    """A cache of a few rows: most CTAs of a one-wave grid get no rows, and a head's pieces
    skip them when they are merged."""
    B, L, hkv, G, d = 1, 1, 4, 4, 128
    c = build_cache(B, L, hkv, G, d, np.array(lens), reserve=2, dtype="bf16", seed=13)
    check(c, B, L, hkv, G, d, "bf16", append=True)
    c = build_cache(B, L, hkv, G, d, np.array(lens), reserve=2, dtype="bf16", seed=14)
    check(c, B, L, hkv, G, d, "bf16", append=False)


def test_decode_repeated_steps_match_single_oracle_run():
    """Several decode steps in a row (appends accumulate) against the oracle step by step."""
    B, L, hkv, G, d = 1, 1, 4, 4, 128
    lens = np.array([100, 3000, 1, 0])
    c = build_cache(B, L, hkv, G, d, lens, reserve=4, dtype="bf16", seed=7)
    dev = "cuda"
    shape = kv.KvShape.of(batch=B, layers=L, hq=hkv * G, hkv=hkv, d=d, n=100000, w=1, pool=1,
                          dtype="bf16")
    scale = 1.0 / math.sqrt(d)
    kf, vf = c["kf"].to(dev), c["vf"].to(dev)
    cu, lens_d = c["cu"].to(dev), c["lens"].to(dev)
    ws = workspace(kv.KV_OP_DECODE, shape)
    Kf, Vf = np64(c["kf"]), np64(c["vf"])
    ln = c["lens"].numpy().astype(np.int64)
    cu_h = c["cu"].numpy()[0]
    gen = torch.Generator().manual_seed(11)
    for step in range(4):
        q = torch.randn(B, L, hkv * G, d, generator=gen).to(torch.bfloat16)
        kn = torch.randn(B, L, hkv, d, generator=gen).to(torch.bfloat16)
        vn = torch.randn(B, L, hkv, d, generator=gen).to(torch.bfloat16)
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        kv.flat_decode_attn(shape, q.to(dev), kn.to(dev), vn.to(dev), kf, vf, cu, lens_d, scale,
                            out, ws)
        assert kv.kv_check_device_status(ws) == 0
        ref, Kf, Vf, ln = O.flat_decode(np64(q[0, 0]), Kf, Vf, cu_h, ln, scale, np64(kn[0, 0]),
                                        np64(vn[0, 0]))
        got = np64(out[0, 0])
        assert_decode_close(got, ref, "bf16", what="decode step %d" % step)
    np.testing.assert_array_equal(lens_d.cpu().numpy(), ln)


@pytest.mark.parametrize("dtype,d,G", [("bf16", 128, 4), ("f32", 64, 2), ("bf16", 128, 8),
                                        ("bf16", 128, 1)])
def test_decode_heads_at_part_boundaries(dtype, d, G):
    """Head lengths around the part sizes of the kernel that cuts heads into parts (192 rows,
    16 per ring stage): one row short of a part, a whole part, one row over, two parts and
    one over, and one head of hundreds of parts, so that every CTA of the grid takes several
    extra parts and the last part of a head merges more than one round of eight partials."""
    B, L, hkv = 1, 2, 8
    lens = np.array([191, 192, 193, 384, 385, 0, 1, 60000,
                     127, 128, 129, 255, 256, 2000, 3, 12345])
    c = build_cache(B, L, hkv, G, d, lens, reserve=2, dtype=dtype, seed=21)
    check(c, B, L, hkv, G, d, dtype, append=True)


@pytest.mark.parametrize("dtype,d,G", [("bf16", 128, 4), ("f32", 64, 2)])
def test_decode_one_fill_first_parts(dtype, d, G):
    """256 heads, most shorter than one ring fill (192 rows) and a few around one to three
    fills, so that their extra parts all find an idle CTA with part 0 at a single fill: the
    kernel that cuts heads into parts then keeps one fill in part 0 and shortens the extra part
    next to it by the rows that fill already holds."""
    B, L, hkv = 1, 32, 8
    rng = np.random.default_rng(37)
    H = B * L * hkv
    lens = rng.integers(1, 190, H)
    edge = [190, 191, 192, 193, 254, 255, 256, 257, 320, 382, 383, 384, 385, 446, 447, 448,
            449, 574, 575, 576, 577, 640, 0]
    lens[rng.choice(H, len(edge), replace=False)] = edge
    c = build_cache(B, L, hkv, G, d, lens, reserve=2, dtype=dtype, seed=38)
    check(c, B, L, hkv, G, d, dtype, append=True)


def test_decode_most_heads_the_parts_kernel_takes():
    """512 heads (the most the kernel that cuts heads into parts takes) of uneven lengths: more
    heads than CTAs of one wave, so the heads' own CTAs take extra parts too."""
    B, L, hkv, G, d = 2, 32, 8, 4, 128
    rng = np.random.default_rng(23)
    H = B * L * hkv
    lens = np.minimum(rng.lognormal(5.0, 1.0, H).astype(np.int64), 5000)
    c = build_cache(B, L, hkv, G, d, lens, reserve=1, dtype="bf16", seed=24)
    check(c, B, L, hkv, G, d, "bf16", append=True)


def test_decode_few_idle_ctas_long_first_parts():
    """296 heads (a few CTAs of a two-per-SM launch left over) of skewed lengths: the kernel
    that cuts heads into parts has to take longer first parts, streamed through its rings,
    before the extra parts of the longest heads fit the idle CTAs."""
    B, L, hkv, G, d = 1, 37, 8, 4, 128
    rng = np.random.default_rng(29)
    H = B * L * hkv
    lens = np.minimum(rng.lognormal(np.log(200.0), 0.6, H).astype(np.int64), 3000)
    c = build_cache(B, L, hkv, G, d, lens, reserve=2, dtype="bf16", seed=30)
    check(c, B, L, hkv, G, d, "bf16", append=True)


def test_decode_parts_lengths_bumped_at_the_end():
    """A head of 480K rows: more extra parts than eight per CTA, so the kernel that cuts heads
    into parts keeps every CTA's extra-part lengths unread until it needs them and bumps the
    lengths after the last CTA is done (the other cases bump them right after the scan)."""
    B, L, hkv, G, d = 1, 1, 2, 2, 64
    lens = np.array([480000, 5])
    c = build_cache(B, L, hkv, G, d, lens, reserve=2, dtype="f32", seed=31)
    check(c, B, L, hkv, G, d, "f32", append=True)


@pytest.mark.parametrize("append", [True, False])
def test_decode_heads_around_whole_extra_parts(append):
    """Lengths around part 0's smallest size (384 rows) plus whole extra parts of 192: a head
    is split only where at least one whole extra part fits, part 0 keeping the remainder."""
    B, L, hkv, G, d = 1, 2, 8, 4, 128
    lens = np.array([383, 384, 385, 575, 576, 577, 767, 768,
                     769, 959, 960, 961, 10, 0, 1000, 1151])
    c = build_cache(B, L, hkv, G, d, lens, reserve=2, dtype="bf16", seed=41)
    check(c, B, L, hkv, G, d, "bf16", append=append)
