"""GPU parity of quantize-on-write (kvq_append) and dequant (kvq_dequant) against
the CPU oracle: bit-exact for every cache byte and every INT8 / INT4 row scale."""
import numpy as np
import pytest
import torch

import fp8_int8_quantized_gb300 as kvq
import oracle
from fp8_int8_quantized_gb300 import workloads as W
from tests.gpu_util import ORACLE_FMT, DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.build()
    torch.cuda.init()


def gpu_cache_to_oracle(c: kvq.KVCache) -> oracle.Cache:
    return oracle.Cache(c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim, c.fmt,
                        k_codes=c.k_codes.cpu().numpy(), v_codes=c.v_codes.cpu().numpy(),
                        k_scales=None if c.k_scales is None else c.k_scales.cpu().numpy(),
                        v_scales=None if c.v_scales is None else c.v_scales.cpu().numpy(),
                        group=c.group_size)


def run_both(k, v, slots, NB, Hkv, BS, D, fmt, scale, group=0):
    dev = torch.device("cuda")
    c = kvq.KVCache(NB, Hkv, BS, D, fmt, dev, fill=0xA5, group_size=group)
    st = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=dev)
    kvq.append(k.to(dev), v.to(dev), c, slots.to(dev), st)
    torch.cuda.synchronize()
    ref = oracle.Cache(NB, Hkv, BS, D, ORACLE_FMT[fmt] if isinstance(fmt, str) else fmt, group=group)
    if c.k_scales is not None:
        ref.k_scales[:] = 0
        ref.v_scales[:] = 0
    oracle.append(k.numpy(), v.numpy(), slots.numpy(), ref, scale)
    return c, ref


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scale", [None, 0.0123, 3.7, 1.0 / 448.0, 0.125, 1e-6])
def test_encoder_every_fp16_pattern(fmt, scale):
    """All 65536 fp16 bit patterns (NaN, Inf, subnormals included) through the
    hardware conversion, after division by several scales."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    k = bits.view(torch.float16).reshape(512, 1, 128).clone()
    v = bits.flip(0).view(torch.float16).reshape(512, 1, 128).clone()
    slots = torch.arange(512, dtype=torch.int64)
    c, ref = run_both(k, v, slots, 32, 1, 16, 128, fmt, scale)
    gk, gv = c.k_codes.cpu().numpy(), c.v_codes.cpu().numpy()
    x = k.float().reshape(32, 1, 16, 128).numpy()
    nan = np.isnan(x)
    bad = (gk != ref.k_codes) & ~nan
    assert not bad.any(), (np.flatnonzero(bad)[:8], gk[bad][:8], ref.k_codes[bad][:8])
    assert np.array_equal(gv[~np.isnan(v.float().reshape(32, 1, 16, 128).numpy())],
                          ref.v_codes[~np.isnan(v.float().reshape(32, 1, 16, 128).numpy())])
    # NaN inputs: both sides give a NaN code of the format
    tab = oracle.fp8_decode_table(ORACLE_FMT[fmt])
    assert np.isnan(tab[gk[nan]]).all()
    assert (ref.k_codes[nan] == 0x7F).all()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scale", [None, 0.0123, 3.7, -0.75, 1.0 / 448.0, 1e-6, 0.2409319132566452, 3e-33, 0.125])
def test_encoder_every_fp16_pattern_large_append(fmt, scale):
    """Appends large enough for the bulk kernel (2^22 values or more; it
    quantizes from the reciprocal of the scale and takes the IEEE division near
    the codes' midpoints): 64 copies of every fp16 bit pattern in shuffled
    slots, bit-exact against the oracle; a negative scale, a power of two, a
    scale whose reciprocal would lose precision (division for every value) and
    the 70B workload's calibration scale included."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.float16)
    g = torch.Generator().manual_seed(17)
    k = bits.repeat(64)[torch.randperm(64 * 65536, generator=g)].reshape(-1, 1, 128).clone()
    v = bits.repeat(64).flip(0).reshape(-1, 1, 128).clone()
    T = k.shape[0]
    slots = torch.randperm(T + 100, generator=g)[:T].to(torch.int64)
    NB = (T + 100 + 15) // 16
    c, ref = run_both(k, v, slots, NB, 1, 16, 128, fmt, scale)
    gk, gv = c.k_codes.cpu().numpy(), c.v_codes.cpu().numpy()
    tab = oracle.fp8_decode_table(ORACLE_FMT[fmt])
    for got, want in ((gk, ref.k_codes), (gv, ref.v_codes)):
        nan = np.isnan(tab[want]) & (want != 0xA5)
        assert np.array_equal(got[~nan], want[~nan])
        assert np.isnan(tab[got[nan]]).all()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scale", [0.0173, 0.2409319132566452, 3.7, 1.0 / 448.0])
def test_large_append_near_code_midpoints(fmt, scale):
    """Inputs whose quotients x / s sit on or next to the midpoints between
    adjacent codes (where the reciprocal's quotient may round the other way):
    for every midpoint m of the format's positive values, the fp16 values
    nearest m * s and their fp16 neighbours two steps either way, both signs,
    repeated past 2^22 values so that the bulk kernel runs; bit-exact against
    the oracle's division."""
    tab = oracle.fp8_decode_table(ORACLE_FMT[fmt]).astype(np.float64)
    pos = np.unique(tab[np.isfinite(tab) & (tab > 0)])
    mids = (pos[:-1] + pos[1:]) / 2
    centre = np.minimum(mids * scale, 65504.0).astype(np.float16).view(np.int16).astype(np.int32)
    cand = np.concatenate([centre + d for d in range(-2, 3)])
    cand = cand[(cand > 0) & (cand < 0x7C00)].astype(np.int16).view(np.float16)
    vals = np.concatenate([cand, -cand]).astype(np.float16)
    reps = (1 << 22) // vals.size + 1
    g = torch.Generator().manual_seed(23)
    flat = torch.from_numpy(np.tile(vals, reps))
    flat = flat[torch.randperm(flat.numel(), generator=g)]
    n = flat.numel() // 128 * 128
    k = flat[:n].reshape(-1, 1, 128).clone()
    v = flat[:n].flip(0).reshape(-1, 1, 128).clone()
    T = k.shape[0]
    slots = torch.arange(T, dtype=torch.int64)
    c, ref = run_both(k, v, slots, (T + 15) // 16, 1, 16, 128, fmt, scale)
    assert np.array_equal(c.k_codes.cpu().numpy(), ref.k_codes)
    assert np.array_equal(c.v_codes.cpu().numpy(), ref.v_codes)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("Hkv,D,BS", [(3, 128, 16), (5, 64, 64), (40, 128, 32), (1, 64, 16)])
def test_large_append_bit_exact_heads_and_blocks(fmt, Hkv, D, BS):
    """The code-table kernel (appends of 2^22 values or more) on random rows
    for several kv-head counts -- its row-to-token division is a multiply-high
    -- head sizes and block sizes, with skipped slots and a ragged last pass."""
    g = torch.Generator().manual_seed(Hkv * 1000 + D + BS)
    T = (1 << 22) // (Hkv * D) + 37
    k = (torch.randn((T, Hkv, D), generator=g) * 2).to(torch.float16)
    v = (torch.randn((T, Hkv, D), generator=g) * 2).to(torch.float16)
    NB = (T + 200 + BS - 1) // BS
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    slots[::13] = -1
    scale = 0.0173 if fmt == "e4m3" else None
    c, ref = run_both(k, v, slots, NB, Hkv, BS, D, fmt, scale)
    assert np.array_equal(c.k_codes.cpu().numpy(), ref.k_codes)
    assert np.array_equal(c.v_codes.cpu().numpy(), ref.v_codes)
    assert kvq.device_error_check()[0] == 0


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "int8", "int4"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("BS", [16, 32, 64])
def test_append_bit_exact(fmt, D, BS):
    g = torch.Generator().manual_seed(D * 7 + BS + len(fmt))
    Hkv, NB, T = 3, 9, 70
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.float16)
    v = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.float16)
    k[5, 1] = 0                     # an all-zero INT8 row
    v[7, 2, 3] = 60000.0            # saturates E4M3
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    slots[::9] = -1
    scale = None if fmt != "e4m3" else 0.02
    c, ref = run_both(k, v, slots, NB, Hkv, BS, D, fmt, scale)
    assert np.array_equal(c.k_codes.cpu().numpy(), ref.k_codes)
    assert np.array_equal(c.v_codes.cpu().numpy(), ref.v_codes)
    if fmt in ("int8", "int4"):
        assert np.array_equal(c.k_scales.cpu().numpy().view(np.uint32), ref.k_scales.view(np.uint32))
        assert np.array_equal(c.v_scales.cpu().numpy().view(np.uint32), ref.v_scales.view(np.uint32))
    st, _ = kvq.device_error_check()
    assert st == 0


def test_append_out_of_range_slot_reported_not_written():
    k = torch.randn((4, 2, 64)).to(torch.float16)
    slots = torch.tensor([0, 5, 10 ** 6, 3], dtype=torch.int64)
    c, ref = run_both(k, k.clone(), torch.tensor([0, 5, -1, 3], dtype=torch.int64), 2, 2, 16, 64, "e4m3", None)
    c2 = kvq.KVCache(2, 2, 16, 64, "e4m3", "cuda", fill=0xA5)
    kvq.append(k.cuda(), k.cuda(), c2, slots.cuda())
    st, detail = kvq.device_error_check()
    assert st == 4  # KVQ_ERR_OUT_OF_RANGE
    assert detail == 10 ** 6
    assert np.array_equal(c2.k_codes.cpu().numpy(), ref.k_codes)
    assert kvq.device_error_check()[0] == 0        # cleared


def test_append_empty_and_validation():
    c = kvq.KVCache(2, 2, 16, 64, "e4m3", "cuda", fill=0xA5)
    e = torch.empty((0, 2, 64), dtype=torch.float16, device="cuda")
    kvq.append(e, e, c, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert (c.k_codes == 0xA5).all()
    with pytest.raises(kvq.KvqError) as ei:
        c.fmt = kvq.E5M2
        d = c.desc()
        d.fmt = kvq.E4M3
        import ctypes
        st = kvq.lib().kvq_append(e.data_ptr(), e.data_ptr(), ctypes.byref(d), 0, 1, None, kvq.E5M2, None)
        kvq._check(st, "kvq_append")
    assert ei.value.status == 1


@pytest.mark.parametrize("fmt", ["int8", "int4"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ng", [2, 4])
def test_append_groups_bit_exact(fmt, D, ng):
    """Group quantization: every code and every group scale bit-exact, with an
    outlier channel, an all-zero group beside non-zero ones and an all-zero row."""
    g = torch.Generator().manual_seed(D * 3 + ng + len(fmt))
    Hkv, NB, BS, T = 3, 7, 16, 90
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.float16)
    v = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.float16)
    k[:, 1, 5] *= 20
    v[2, 0, :D // ng] = 0
    k[6, 2] = 0
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    slots[::11] = -1
    c, ref = run_both(k, v, slots, NB, Hkv, BS, D, fmt, None, group=D // ng)
    assert c.k_scales.shape == (NB, Hkv, BS, ng)
    assert np.array_equal(c.k_codes.cpu().numpy(), ref.k_codes)
    assert np.array_equal(c.v_codes.cpu().numpy(), ref.v_codes)
    assert np.array_equal(c.k_scales.cpu().numpy().view(np.uint32), ref.k_scales.view(np.uint32))
    assert np.array_equal(c.v_scales.cpu().numpy().view(np.uint32), ref.v_scales.view(np.uint32))
    ok, ov = kvq.dequant(c, slots.clamp(min=0).cuda())
    rk, rv = oracle.dequant(ref, slots.clamp(min=0).numpy())
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv.view(np.uint32))
    assert kvq.device_error_check()[0] == 0


@pytest.mark.parametrize("fmt,group", [("int8", 0), ("int4", 0), ("int8", 32), ("int4", 64)])
def test_append_rounding_ties_and_bulk_rows_bit_exact(fmt, group):
    """INT8 / INT4 codes are rint(fl32(x / s)), ties to even.  Rows whose scale
    is a power of two make x / s exactly k + 0.5 (ties), or one fp16 step off
    it (near-ties); then a bulk append of 24000 random rows with x20 outlier
    channels (about 3000 values whose quotient lies within 2^-14 of a
    half-integer).  Every code and scale bit-exact against the oracle."""
    qmax = 127 if fmt == "int8" else 7
    Hkv, D = 2, 128
    ties = []
    for e in (-3, 0, 2):                          # s = 2^e exactly: amax = qmax * 2^e
        s = 2.0 ** e
        row = torch.zeros(D, dtype=torch.float64)
        row[0] = qmax * s
        k = torch.arange(-qmax, qmax)              # k + 0.5 for k in [-qmax, qmax - 1]
        n = min(D - 1, k.numel())
        row[1:1 + n] = (k[:n] + 0.5) * s
        ties.append(row)
        near = row.clone().to(torch.float16)
        nb = near.view(torch.int16)
        nb[1:] += 1                                # the next fp16 value away from zero
        ties.append(near.double())
    sub = torch.randn(D, dtype=torch.float64, generator=torch.Generator().manual_seed(5)) * 2e-6
    ties.append(sub)                               # a row of fp16 subnormals (a tiny scale)
    t = torch.stack(ties).to(torch.float16)        # [rows][D]
    assert (t[-1].abs() < 6.1e-5).all() and t[-1].any()
    kt = t[:, None, :].repeat(1, Hkv, 1)
    assert (kt.double()[:, 0, 1:1 + 10] / 2.0 ** -3).fmod(1).abs().ne(0).any()   # not all integers
    g = torch.Generator().manual_seed(len(fmt) + group)
    T = 24000
    kb = torch.randn((T, Hkv, D), generator=g) * 2
    vb = torch.randn((T, Hkv, D), generator=g) * 2
    kb[:, :, 7] *= 20
    vb[:, 1, 100] *= 20
    k = torch.cat([kt, kb.to(torch.float16)])
    v = torch.cat([kt.flip(2), vb.to(torch.float16)])
    NB, BS = (k.shape[0] + 15) // 16, 16
    slots = torch.randperm(NB * BS, generator=g)[:k.shape[0]].to(torch.int64)
    c, ref = run_both(k, v, slots, NB, Hkv, BS, D, fmt, None, group=group)
    assert np.array_equal(c.k_codes.cpu().numpy(), ref.k_codes)
    assert np.array_equal(c.v_codes.cpu().numpy(), ref.v_codes)
    assert np.array_equal(c.k_scales.cpu().numpy().view(np.uint32), ref.k_scales.view(np.uint32))
    assert np.array_equal(c.v_scales.cpu().numpy().view(np.uint32), ref.v_scales.view(np.uint32))
    assert kvq.device_error_check()[0] == 0


@pytest.mark.parametrize("name", ["llama2-7b", "llama3-8b", "llama2-13b-int8", "llama2-13b-int4", "llama3-70b",
                                  "llama2-13b-int4-g32", "llama3-70b-int8-g32", "llama3-70b-int4-g32"])
def test_append_full_size_sampled(name):
    """The workloads' own append launches (their full windows), checked on a
    seeded sample of tokens against the oracle."""
    wl = W.WORKLOADS[name]
    lay = W.Layout(wl)
    win = (wl.ctx - wl.append_chunk, wl.ctx) if wl.append_chunk else W.chunk_positions(wl, 1 << 19)[0]
    dev = torch.device("cuda")
    k, v = W.kv_tokens(wl, *win, device=dev)
    slots = lay.slots(*win).to(dev)
    scale_v = W.calibration_scale(wl, k, v)
    scale = None if scale_v is None else torch.tensor([scale_v], dtype=torch.float32, device=dev)
    c = kvq.KVCache(lay.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim, wl.fmt, dev, fill=0xA5,
                    group_size=wl.quant_group)
    kvq.append(k, v, c, slots, scale)
    torch.cuda.synchronize()
    assert kvq.device_error_check()[0] == 0
    gen = torch.Generator().manual_seed(7)
    valid = torch.nonzero(slots.cpu() >= 0).flatten()
    pick = valid[torch.randperm(valid.numel(), generator=gen)[:256]]
    s = slots.cpu()[pick]
    pd = pick.to(dev)
    ks, vs = k[pd].cpu(), v[pd].cpu()
    ref = oracle.Cache(len(pick) // wl.block_size + 1, wl.num_kv_heads, wl.block_size, wl.head_dim,
                       ORACLE_FMT[wl.fmt], group=wl.quant_group)
    oracle.append(ks.numpy(), vs.numpy(), np.arange(len(pick), dtype=np.int64), ref, scale_v)
    bs = wl.block_size
    blk, off = (s // bs).to(dev), (s % bs).to(dev)
    gk = c.k_codes[blk, :, off].cpu().numpy()
    gv = c.v_codes[blk, :, off].cpu().numpy()
    i = np.arange(len(pick))
    assert np.array_equal(gk, ref.k_codes[i // bs, :, i % bs])
    assert np.array_equal(gv, ref.v_codes[i // bs, :, i % bs])
    if wl.fmt in ("int8", "int4"):
        assert np.array_equal(c.k_scales[blk, :, off].cpu().numpy(), ref.k_scales[i // bs, :, i % bs])
        assert np.array_equal(c.v_scales[blk, :, off].cpu().numpy(), ref.v_scales[i // bs, :, i % bs])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "int8", "int4"])
@pytest.mark.parametrize("D", [64, 128])
def test_dequant_bit_exact(fmt, D):
    g = torch.Generator().manual_seed(3 + D)
    Hkv, NB, BS, T = 2, 6, 16, 50
    k = (torch.randn((T, Hkv, D), generator=g) * 5).to(torch.float16)
    v = (torch.randn((T, Hkv, D), generator=g) * 5).to(torch.float16)
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    scale = 0.05 if fmt not in ("int8", "int4") else None
    c, ref = run_both(k, v, slots, NB, Hkv, BS, D, fmt, scale)
    st = None if scale is None else torch.tensor([scale], dtype=torch.float32, device="cuda")
    ok, ov = kvq.dequant(c, slots.cuda(), st)
    rk, rv = oracle.dequant(ref, slots.numpy(), scale)
    assert np.array_equal(ok.cpu().numpy().view(np.uint32), rk.view(np.uint32))
    assert np.array_equal(ov.cpu().numpy().view(np.uint32), rv.view(np.uint32))
