"""The stochastic verifier's arithmetic contract, primitive by primitive, on
the GPU against the CPU oracle, bit for bit.

Every stochastic decision rests on the kernel's own exp E, its fixed-point
weights FX and their accumulators, and its residual division agreeing with
the oracle's independent implementation of the same contract exactly.  The
parity tests see these only through accept/reject outcomes; here the device
functions run over arrays (spec_selftest_exp / _fx / _resid, which call the
verifier's own device code) and every result is compared:
  * E, scalar and two-lane, over EVERY fp32 in [-87, 0] (1 118 699 521
    values) plus the region below -87, -inf and NaN (which give 0);
  * FX over every fp32 in [0, 2) (2^30 values); the scalar accumulator on
    one-entry segments and the two-lane accumulator on pairs over the same
    range; both accumulators on random 510-entry segments mixing values
    below, at and above 1;
  * one residual step max(d / Z - q, 0) by IEEE division and by the
    Markstein sequences (scalar and two-lane) on 16.7M random entries of the
    verifier's domain (d in [0, 1], Z = fp32(S) * 2^-46).
The device outputs are compared with the oracle on the host (for FX, the two
accumulators are compared on the device with the FX values already checked
against the oracle, which keeps the copies to one per chunk)."""
import ctypes
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle as O
import tree_speculative_verification_spec_gb300 as S

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26
POOL = 8


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tree_speculative_verification_spec_gb300 import build
    build.build()
    S.lib()
    O.lib()


def _oracle_parallel(fn, *arrays, out_dtype):
    """Run an oracle array helper over equal slices of its inputs on threads
    (ctypes releases the GIL during the call)."""
    n = arrays[0].size
    parts = np.linspace(0, n, POOL + 1).astype(np.int64)
    outs = [None] * POOL

    def one(k):
        sl = slice(parts[k], parts[k + 1])
        outs[k] = fn(*[a[sl] for a in arrays])

    with ThreadPoolExecutor(POOL) as ex:
        list(ex.map(one, range(POOL)))
    res = np.concatenate(outs)
    assert res.dtype == out_dtype
    return res


def _exp_range(first, count):
    """Compare E over bit patterns first .. first + count - 1 (chunked)."""
    done = 0
    while done < count:
        n = min(CHUNK, count - done)
        start = (first + done) & 0xFFFFFFFF
        es = torch.empty(n, dtype=torch.float32, device="cuda")
        ep = torch.empty(n, dtype=torch.float32, device="cuda")
        S.spec_selftest_exp(start, n, es, ep)
        if start + n <= 1 << 32:
            bits = np.arange(start, start + n, dtype=np.uint32)
        else:  # the patterns wrap modulo 2^32
            bits = (np.arange(n, dtype=np.uint64) + np.uint64(start)).astype(np.uint32)
        ref = _oracle_parallel(O.canon_exp, bits.view(np.float32), out_dtype=np.float32).view(np.uint32)
        for name, t in (("scalar", es), ("two-lane", ep)):
            got = t.cpu().numpy().view(np.uint32)
            bad = np.flatnonzero(got != ref)
            assert bad.size == 0, (name, int(bad.size), [(hex(int(bits[i])), float(bits[i:i + 1].view(np.float32)[0]),
                                                         hex(int(got[i])), hex(int(ref[i]))) for i in bad[:6]])
        done += n


def test_exp_every_float_in_minus87_to_0():
    first, last = 0x80000000, int(np.float32(-87.0).view(np.uint32))  # -0.0 .. -87.0
    _exp_range(first, last - first + 1)
    _exp_range(0x00000000, 1)  # +0.0


def test_exp_below_minus87_and_specials_is_zero():
    _exp_range(int(np.float32(-87.0).view(np.uint32)) + 1, 1 << 20)  # just below -87
    for bits in (0xFF800000, 0xFFC00000, 0x7FC00000, 0xC2B00000, 0xF0000000):  # -inf, NaNs, -88, -1.6e29
        _exp_range(bits, 1)


def test_fx_every_float_in_0_to_2_and_both_accumulators():
    total = 1 << 30  # bit patterns 0x00000000 .. 0x3FFFFFFF: every fp32 in [0, 2)
    for start in range(0, total, CHUNK):
        n = CHUNK
        v = torch.arange(start, start + n, dtype=torch.int32, device="cuda").view(torch.float32)
        fx = torch.empty(n, dtype=torch.int64, device="cuda")
        one = torch.empty(n, dtype=torch.int64, device="cuda")
        pair = torch.empty(n // 2, dtype=torch.int64, device="cuda")
        S.spec_selftest_fx(v, 1, fx_out=fx, seg_scalar=one)
        S.spec_selftest_fx(v, 2, seg_pair=pair)
        # per entry: the scalar accumulator holds exactly fx; per pair: the
        # two-lane accumulator holds exactly the sum of the pair's fx (device)
        assert torch.equal(one, fx), start
        assert torch.equal(pair, fx[0::2] + fx[1::2]), start
        got = fx.cpu().numpy().view(np.uint64)
        vals = np.arange(start, start + n, dtype=np.uint32).view(np.float32)
        ref = _oracle_parallel(O.fx_array, vals, out_dtype=np.uint64)
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, [(hex(start + int(i)), int(got[i]), int(ref[i])) for i in bad[:5]]


def test_fx_accumulators_on_random_segments():
    rng = np.random.default_rng(3)
    seg, nseg = 510, 20000
    n = seg * nseg
    kind = rng.integers(0, 6, size=n)
    v = np.where(kind == 0, rng.random(n), 0.0)
    v = np.where(kind == 1, 1.0, v)
    v = np.where(kind == 2, 1.0 + rng.random(n), v)                   # (1, 2): the 64-bit path
    v = np.where(kind == 3, rng.random(n) * 2.0 ** -40, v)            # a few fixed-point units
    v = np.where(kind == 4, 2.0 ** -rng.integers(0, 149, size=n), v)  # powers of two, subnormals
    v = np.where(kind == 5, np.nextafter(np.float32(1.0), np.float32(0.0)), v)
    v = v.astype(np.float32)
    v[rng.integers(0, n, size=n // 50)] = 0.0
    dv = torch.from_numpy(v).cuda()
    s1 = torch.empty(nseg, dtype=torch.int64, device="cuda")
    s2 = torch.empty(nseg, dtype=torch.int64, device="cuda")
    S.spec_selftest_fx(dv, seg, seg_scalar=s1, seg_pair=s2)
    ref = O.fx_array(v).reshape(nseg, seg).sum(axis=1, dtype=np.uint64)
    assert np.array_equal(s1.cpu().numpy().view(np.uint64), ref)
    assert np.array_equal(s2.cpu().numpy().view(np.uint64), ref)


def test_residual_step_division_and_markstein_sequences():
    rng = np.random.default_rng(11)
    n = 1 << 24
    e = rng.integers(0, 130, size=n)
    d = (2.0 ** -e.astype(np.float64) * (1.0 + rng.random(n))).clip(0, 1).astype(np.float32)  # [2^-129, 1]
    d[rng.integers(0, n, size=n // 64)] = 0.0
    d[rng.integers(0, n, size=n // 64)] = 1.0
    q = (rng.random(n) ** 4).astype(np.float32)
    q[rng.integers(0, n, size=n // 64)] = 0.0
    Sx = rng.integers(1, 2 ** 63 - 1, size=n // 2, dtype=np.int64) >> rng.integers(0, 63, size=n // 2)
    Zp = (np.maximum(Sx, 1).astype(np.float32) * np.float32(2.0 ** -46)).astype(np.float32)
    # normalisers at and next to powers of two, within [2^-46, 2^17)
    edge = [np.float32(2.0 ** k) for k in range(-46, 17)]
    edge += [np.nextafter(np.float32(2.0 ** k), np.float32(np.inf)) for k in range(-46, 17)]
    edge += [np.nextafter(np.float32(2.0 ** k), np.float32(-np.inf)) for k in range(-45, 17)]
    Zp[: 64 * len(edge)] = np.tile(np.array(edge, np.float32), 64)
    ref = O.resid_step(d, q, Zp)
    dd, dq, dz = (torch.from_numpy(a).cuda() for a in (d, q, Zp))
    outs = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    S.spec_selftest_resid(dd, dq, dz, r_div=outs[0], r_markstein=outs[1], r_pair=outs[2])
    for name, o in zip(("division", "markstein", "pair"), outs):
        got = o.cpu().numpy().view(np.uint32)
        bad = np.flatnonzero(got != ref.view(np.uint32))
        assert bad.size == 0, (name, [(float(d[i]), float(Zp[i // 2]), float(q[i])) for i in bad[:5]])


def test_selftest_argument_checks():
    L = S.lib()
    assert L.spec_selftest_exp(0, -1, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_exp(0, 4, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_fx(None, 6, 4, None, None, None, None) == S.SPEC_ERR_INVALID_ARG  # n % seg
    # an odd segment with the two-lane output is refused before any pointer is used
    assert L.spec_selftest_fx(None, 9, 3, None, None, ctypes.c_void_p(256), None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_fx(None, 1022, 511, None, None, None, None) == S.SPEC_ERR_INVALID_ARG
    assert L.spec_selftest_resid(None, None, None, 4, None, None, None, None) == S.SPEC_ERR_INVALID_ARG
