"""Pins of the CPU oracle to things other than itself.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with what the method's description and plain mathematics fix:

* hand-worked goldens (tests/golden/*.txt, each with its derivation);
* exact rational re-derivation of every rounding on random rows;
* invariants (code range, absmax element -> +-127, round-trip error <= s/2);
* special cases (static scale 1 on integers is the identity; an identity block
  table with one block per sequence is contiguous per-sequence quantisation);
* a brute-force placement model on random tiny block tables with a sentinel
  pool.

``test_oracle_pins`` runs them on the committed oracle; ``test_oracle_mutations``
runs them on copies of the oracle with planted mistakes and requires that at
least one pin rejects each copy.
"""
from fractions import Fraction as F

import numpy as np

import _exact as ex
import _golden


def _bf16_bits_exact(decimals):
    """Decimal strings -> bf16 bits, asserting each value is exact in bf16."""
    out = []
    for s in decimals:
        v = F(s) if s not in ("-0", "-0.0") else F(0)
        if v == 0:
            out.append(0x8000 if s.startswith("-") else 0)
            continue
        out.append(ex.bf16_bits_of(v))
    return np.array(out, np.uint16)


def _bits_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def _f32_bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ---- goldens -------------------------------------------------------------------

def pin_quantize_goldens(orc):
    for c in _golden.quantize_cases():
        H, D = c["heads"], c["head_dim"]
        x = _bf16_bits_exact(c["x"]).reshape(1, H, D)
        if c["mode"] == 0:
            q, s = orc.quantize_rows(0, x)
            got_s = [int(b) for b in _f32_bits(s[0])]
            assert got_s == c["scale_bits"], (c["name"], [hex(b) for b in got_s])
        else:
            static = c["static_bits"].view(np.float32)
            q, _ = orc.quantize_rows(1, x, static)
        assert np.array_equal(q[0].astype(np.int64), c["codes"]), (c["name"], q[0])


def pin_dequant_goldens(orc):
    for q, sbits, expect in _golden.dequant_values():
        s = np.array([sbits], np.uint32).view(np.float32)[0]
        got = orc.dequantize_value(q, s)
        assert got == expect, (q, hex(sbits), hex(got), hex(expect))


def _token_rows_placement(n_tokens, D):
    rows = np.zeros((n_tokens, 1, D), np.float32)
    for t in range(n_tokens):
        rows[t, 0, 0] = 127
        rows[t, 0, 1:] = 10 * t + np.arange(1, D)
    return (rows.view(np.uint32) >> 16).astype(np.uint16)


def pin_placement_golden(orc):
    g = _golden.placement()
    H, D = 1, 16
    bs, NB = g["block_size"], g["num_blocks"]
    n_tok = int(g["cu_q_lens"][-1])
    x = _token_rows_placement(n_tok, D)
    kc = np.full((NB, H, bs, D), 85, np.int8)
    vc = np.full((NB, H, bs, D), 85, np.int8)
    ks = np.full((NB, H, bs), 0.5, np.float32)
    vs = np.full((NB, H, bs), 0.5, np.float32)
    orc.store(0, x, x, kc, vc, ks, vs, g["block_table"], g["cu_q_lens"], g["context_kv_lens"])
    owner = {v: t for t, v in g["expect_slot"].items()}
    for blk in range(NB):
        for slot in range(bs):
            for cache, sc in ((kc, ks), (vc, vs)):
                if (blk, slot) in owner:
                    t = owner[(blk, slot)]
                    want = np.concatenate([[127], 10 * t + np.arange(1, D)])
                    assert np.array_equal(cache[blk, 0, slot].astype(np.int64), want), (blk, slot)
                    assert sc[blk, 0, slot] == 1.0
                else:
                    assert np.all(cache[blk, 0, slot] == 85), (blk, slot)
                    assert sc[blk, 0, slot] == 0.5
    sentinel = 0x422A  # 85 * 0.5 = 42.5
    for gg in g["gathers"]:
        rows = gg.get("out_rows", len(gg["rows"]))
        ko = np.full((rows, H, D), 0xFFFF, np.uint16)
        vo = np.full((rows, H, D), 0xFFFF, np.uint16)
        orc.dequant_gather(0, kc, vc, ks, vs, g["block_table"], gg["context_lengths"],
                           gg.get("offsets"), ko, vo)
        for r, tag in enumerate(gg["rows"]):
            if tag == "F":
                want = np.full(D, 0xFFFF, np.uint16)
            elif tag == "S":
                want = np.full(D, sentinel, np.uint16)
            else:
                t = int(tag)
                vals = [F(127)] + [F(10 * t + d) for d in range(1, D)]
                want = np.array([ex.bf16_bits_of(v) for v in vals], np.uint16)
            assert np.array_equal(ko[r, 0], want), (r, tag, ko[r, 0])
            assert np.array_equal(vo[r, 0], want), (r, tag)


# ---- exact rational re-derivation ----------------------------------------------

def _random_bf16_rows(rng, n, H, D, spread=True):
    x = rng.standard_normal((n, H, D)).astype(np.float32)
    if spread:
        x *= np.exp2(rng.integers(-6, 7, size=(n, H, 1))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 will do
    return bits


def pin_exact_quantize_random(orc):
    rng = np.random.default_rng(7)
    H, D = 2, 16
    # mode 0, random rows, plus rows whose entries sit at amax/2 (quotients near 63.5)
    x = _random_bf16_rows(rng, 24, H, D)
    amax_bits = rng.integers(0x3F80, 0x4280, size=8).astype(np.uint16)
    for i, a in enumerate(amax_bits):
        x[i, 0, 0] = a
        x[i, 0, 1] = a - 0x0080  # a / 2 (exponent minus one)
        x[i, 0, 2] = (a - 0x0080) | 0x8000
        x[i, 0, 3:] = a - 0x0180  # a / 8, so that a stays the row's max
    q, s = orc.quantize_rows(0, x)
    xf = _bits_to_f32(x)
    for t in range(x.shape[0]):
        for h in range(H):
            row = [F(float(v)) for v in xf[t, h]]
            s_exact = ex.expected_row_scale(row)
            assert F(float(s[t, h])) == s_exact, (t, h)
            for d in range(D):
                assert int(q[t, h, d]) == ex.expected_code(row[d], s_exact), (t, h, d)
    # mode 1, random static scales over a wide range (saturating and not)
    static = np.exp(rng.uniform(np.log(0.003), np.log(2.0), size=(H, D))).astype(np.float32)
    q1, _ = orc.quantize_rows(1, x, static)
    for t in range(x.shape[0]):
        for h in range(H):
            for d in range(D):
                want = ex.expected_code(F(float(xf[t, h, d])), F(float(static[h, d])))
                assert int(q1[t, h, d]) == want, (t, h, d)
    # mode 2, one scale per row (the row's block scale), zero included
    per_row = np.exp(rng.uniform(np.log(0.003), np.log(2.0), size=(x.shape[0], H))).astype(np.float32)
    per_row[3, 1] = 0.0
    q2, s2 = orc.quantize_rows(2, x, per_row)
    assert s2 is None
    for t in range(x.shape[0]):
        for h in range(H):
            for d in range(D):
                want = ex.expected_code(F(float(xf[t, h, d])), F(float(per_row[t, h])))
                assert int(q2[t, h, d]) == want, (t, h, d)


def pin_exact_dequant_random(orc):
    rng = np.random.default_rng(11)
    qs = rng.integers(-127, 128, size=400)
    ss = np.exp(rng.uniform(np.log(1e-4), np.log(4.0), size=400)).astype(np.float32)
    # scales with long significands next to bf16 midpoints as well
    ss[:50] = (np.float32(1) + rng.integers(0, 1 << 23, size=50).astype(np.float32) * np.float32(2.0 ** -23))
    for q, s in zip(qs, ss):
        got = orc.dequantize_value(int(q), s)
        want = ex.expected_dequant_bits(int(q), F(float(s)))
        assert got == want, (int(q), float(s), hex(got), hex(want))


# ---- invariants and special cases ------------------------------------------------

def pin_invariants(orc):
    rng = np.random.default_rng(3)
    H, D = 4, 64
    x = _random_bf16_rows(rng, 64, H, D)
    x[5, 1, :] = 0  # an all-zero row
    q, s = orc.quantize_rows(0, x)
    xf = _bits_to_f32(x).astype(np.float64)
    assert q.min() >= -127 and q.max() <= 127
    amax = np.abs(xf).max(axis=2)
    for t in range(x.shape[0]):
        for h in range(H):
            if amax[t, h] == 0:
                assert s[t, h] == 0 and np.all(q[t, h] == 0)
                continue
            at = np.abs(xf[t, h]) == amax[t, h]
            assert np.all(np.abs(q[t, h][at]) == 127), (t, h)
            assert np.all(np.sign(q[t, h][at]) == np.sign(xf[t, h][at]))
    # round trip: |q s - x| <= s (1/2 + 2^-18) (the fp32 quotient is within
    # half an ulp of x/s, and the ulp is at most 2^-17 below 128)
    sf = s.astype(np.float64)[:, :, None]
    err = np.abs(q.astype(np.float64) * sf - xf)
    assert np.all(err <= sf * (0.5 + 2.0 ** -18)), float((err - sf / 2).max())
    # the dequantised bf16 value adds at most half a bf16 ulp of the product
    NB, bs = 16, 4
    kc = np.zeros((NB, H, bs, D), np.int8)
    ks = np.zeros((NB, H, bs), np.float32)
    kc[:, :, :, :] = q.reshape(NB, bs, H, D).transpose(0, 2, 1, 3)
    ks[:, :, :] = s.reshape(NB, bs, H).transpose(0, 2, 1)
    bt = np.arange(NB, dtype=np.int32).reshape(1, NB)
    ko, vo = orc.dequant_gather(0, kc, kc, ks, ks, bt, np.array([NB * bs], np.int32))
    back = _bits_to_f32(ko).astype(np.float64)
    prod = q.astype(np.float64) * sf
    assert np.all(np.abs(back - prod) <= np.abs(prod) * (2.0 ** -8 + 2.0 ** -23))
    assert np.all(np.abs(back - xf) <= sf * (0.5 + 2.0 ** -18) + np.abs(prod) * (2.0 ** -8 + 2.0 ** -23))
    # static scale 1 on integer inputs is the identity
    ints = rng.integers(-127, 128, size=(8, H, D)).astype(np.float32)
    xb = (ints.view(np.uint32) >> 16).astype(np.uint16)
    q1, _ = orc.quantize_rows(1, xb, np.ones((H, D), np.float32))
    assert np.array_equal(q1.astype(np.int64), ints.astype(np.int64))


def pin_identity_table(orc):
    """bs >= every context and block_table[b] = [b]: the store is contiguous
    per-sequence quantisation, row for row."""
    rng = np.random.default_rng(5)
    B, H, D, bs = 3, 2, 32, 64
    q_lens = np.array([7, 64, 1], np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    x = _random_bf16_rows(rng, int(cu[-1]), H, D)
    kc = np.full((B, H, bs, D), -5, np.int8)
    vc = kc.copy()
    ks = np.full((B, H, bs), 9.0, np.float32)
    vs = ks.copy()
    bt = np.arange(B, dtype=np.int32).reshape(B, 1)
    orc.store(0, x, x, kc, vc, ks, vs, bt, cu, np.zeros(B, np.int32))
    q, s = orc.quantize_rows(0, x)
    for b in range(B):
        rows = slice(int(cu[b]), int(cu[b + 1]))
        assert np.array_equal(kc[b, :, :q_lens[b]], q[rows].transpose(1, 0, 2))
        assert np.array_equal(ks[b, :, :q_lens[b]], s[rows].T)
        assert np.all(kc[b, :, q_lens[b]:] == -5) and np.all(ks[b, :, q_lens[b]:] == 9.0)


def pin_cumsum(orc):
    assert list(orc.exclusive_cumsum(np.array([3, 0, 5, 2], np.int32))) == [0, 3, 3, 8]
    assert list(orc.exclusive_cumsum(np.array([7], np.int32))) == [0]


# ---- brute-force placement -----------------------------------------------------

def _bruteforce_once(orc, rng, quant_mode, decode_null_cu):
    B = int(rng.integers(1, 5))
    H = int(rng.integers(1, 3))
    D = 16
    bs = int(rng.choice([1, 2, 4, 16]))
    MB = int(rng.integers(1, 5))
    NB = B * MB + int(rng.integers(0, 3))
    cap = MB * bs
    if decode_null_cu:
        ctx_before = rng.integers(0, cap, size=B)
        q_lens = np.ones(B, np.int64)
    else:
        ctx_before = rng.integers(0, cap + 1, size=B)
        q_lens = np.array([rng.integers(0, cap - c + 1) for c in ctx_before])
    perm = rng.permutation(NB).astype(np.int32)
    bt = perm[:B * MB].reshape(B, MB).copy()
    N = int(q_lens.sum())
    x = _random_bf16_rows(rng, N, H, D)
    y = _random_bf16_rows(rng, N, H, D)
    kc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    if quant_mode == 0:
        ks = rng.uniform(0.01, 0.1, size=(NB, H, bs)).astype(np.float32)
        vs = rng.uniform(0.01, 0.1, size=(NB, H, bs)).astype(np.float32)
    elif quant_mode == 1:
        ks = rng.uniform(0.005, 0.05, size=(H, D)).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, size=(H, D)).astype(np.float32)
    else:  # one scale per physical block and head, all distinct
        ks = rng.uniform(0.005, 0.05, size=(NB, H)).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, size=(NB, H)).astype(np.float32)
    kc0, vc0, ks0, vs0 = kc.copy(), vc.copy(), ks.copy(), vs.copy()
    cu = None if decode_null_cu else np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    orc.store(quant_mode, x, y, kc, vc, ks, vs, bt, cu, ctx_before.astype(np.int32))

    # independent logical model: dict (seq, pos) -> token index
    model = {}
    tok = 0
    for b in range(B):
        for i in range(int(q_lens[b])):
            model[(b, int(ctx_before[b]) + i)] = tok
            tok += 1
    phys = {}
    for (b, p), t in model.items():
        phys[(int(bt[b][p // bs]), p % bs)] = t
    if quant_mode == 2:  # each token takes the scale of the physical block it lands in
        tok_blk = np.zeros(N, np.int64)
        for (b, p), t in model.items():
            tok_blk[t] = bt[b][p // bs]
        qx, sx = orc.quantize_rows(2, x, ks0[tok_blk])
        qy, sy = orc.quantize_rows(2, y, vs0[tok_blk])
    else:
        qx, sx = orc.quantize_rows(quant_mode, x, ks0 if quant_mode == 1 else None)
        qy, sy = orc.quantize_rows(quant_mode, y, vs0 if quant_mode == 1 else None)
    for blk in range(NB):
        for slot in range(bs):
            t = phys.get((blk, slot))
            for cache, c0, qq in ((kc, kc0, qx), (vc, vc0, qy)):
                want = c0[blk, :, slot] if t is None else qq[t]
                assert np.array_equal(cache[blk, :, slot], want), (blk, slot, t)
            if quant_mode == 0:
                for sc, s0, ss in ((ks, ks0, sx), (vs, vs0, sy)):
                    want = s0[blk, :, slot] if t is None else ss[t]
                    assert np.array_equal(sc[blk, :, slot], want), (blk, slot, t)
    if quant_mode != 0:  # static scales are read, never written
        assert np.array_equal(ks, ks0) and np.array_equal(vs, vs0)

    # gather: each output row is the dequantised physical row of its position
    ctx_after = (ctx_before + q_lens).astype(np.int32)
    pad = rng.integers(0, 3, size=B)
    offsets = np.concatenate([[0], np.cumsum(ctx_after + pad)[:-1]]).astype(np.int64)
    rows = int((ctx_after + pad).sum()) + 1
    for off in (None, offsets):
        r = int(ctx_after.sum()) if off is None else rows
        ko = np.full((r, H, D), 0xFFFF, np.uint16)
        vo = np.full((r, H, D), 0xFFFF, np.uint16)
        orc.dequant_gather(quant_mode, kc, vc, ks, vs, bt, ctx_after, off, ko, vo)
        base = orc.exclusive_cumsum(ctx_after) if off is None else off
        covered = np.zeros(r, bool)
        for b in range(B):
            for p in range(int(ctx_after[b])):
                blk, slot = int(bt[b][p // bs]), p % bs
                row = int(base[b]) + p
                covered[row] = True
                for out, cache, sc in ((ko, kc, ks), (vo, vc, vs)):
                    for h in range(H):
                        for d in range(0, D, 5):
                            s = (sc[blk, h, slot] if quant_mode == 0 else
                                 sc[h, d] if quant_mode == 1 else sc[blk, h])
                            want = ex.expected_dequant_bits(int(cache[blk, h, slot, d]),
                                                            F(float(s)))
                            assert int(out[row, h, d]) == want, (b, p, h, d)
        assert np.all(ko[~covered] == 0xFFFF) and np.all(vo[~covered] == 0xFFFF)


def pin_placement_bruteforce(orc):
    rng = np.random.default_rng(2024)
    for it in range(24):
        _bruteforce_once(orc, rng, quant_mode=it % 2, decode_null_cu=(it % 6 == 5))
    rng = np.random.default_rng(2025)
    for it in range(12):  # per-block scales
        _bruteforce_once(orc, rng, quant_mode=2, decode_null_cu=(it % 4 == 3))


def pin_per_block_reduces_to_per_channel(orc):
    """One scale for every block and head, c, is the per-channel table filled
    with c: both modes must store and gather the same bits."""
    rng = np.random.default_rng(31)
    B, H, D, bs, MB = 3, 2, 16, 4, 3
    NB = B * MB + 1
    bt = rng.permutation(NB).astype(np.int32)[:B * MB].reshape(B, MB).copy()
    q_lens = np.array([5, 1, 7])
    ctx = np.array([2, 0, 4], np.int32)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    x = _random_bf16_rows(rng, int(q_lens.sum()), H, D)
    y = _random_bf16_rows(rng, int(q_lens.sum()), H, D)
    c = np.float32(0.0173)
    pools = []
    for mode, ks in ((1, np.full((H, D), c, np.float32)), (2, np.full((NB, H), c, np.float32))):
        kc = np.zeros((NB, H, bs, D), np.int8)
        vc = np.zeros((NB, H, bs, D), np.int8)
        orc.store(mode, x, y, kc, vc, ks, ks.copy(), bt, cu, ctx)
        lens = ctx + q_lens.astype(np.int32)
        ko, vo = orc.dequant_gather(mode, kc, vc, ks, ks, bt, lens)
        pools.append((kc, vc, ko, vo))
    for a, b in zip(*pools):
        assert np.array_equal(a, b)


def pin_bounds_errors(orc):
    """A block id outside the pool, or a position beyond the block table, is an
    error, not a silent write."""
    import oracle as _o
    H, D, bs, NB = 1, 16, 4, 2
    x = np.zeros((1, H, D), np.uint16)
    kc = np.zeros((NB, H, bs, D), np.int8)
    ks = np.zeros((NB, H, bs), np.float32)
    for bt, ctx in ((np.array([[5]], np.int32), 0), (np.array([[1]], np.int32), 4)):
        try:
            orc.store(0, x, x, kc, kc.copy(), ks, ks.copy(), bt, np.array([0, 1], np.int32),
                      np.array([ctx], np.int32))
        except _o.OracleError:
            continue
        raise AssertionError("out-of-range store accepted")


# ---- bf16 cache (no quantisation) -----------------------------------------------

def pin_bf16_placement_golden(orc):
    """The hand-worked placement of tests/golden/placement_tiny.txt, with a bf16
    cache: rows land, and are gathered, bit for bit."""
    g = _golden.placement()
    H, D = 1, 16
    bs, NB = g["block_size"], g["num_blocks"]
    n_tok = int(g["cu_q_lens"][-1])
    x = _token_rows_placement(n_tok, D)
    y = x ^ np.uint16(0x0001)  # V rows differ from K rows
    kc = np.full((NB, H, bs, D), 0x1234, np.uint16)
    vc = np.full((NB, H, bs, D), 0x4321, np.uint16)
    orc.store_bf16(x, y, kc, vc, g["block_table"], g["cu_q_lens"], g["context_kv_lens"])
    owner = {v: t for t, v in g["expect_slot"].items()}
    for blk in range(NB):
        for slot in range(bs):
            t = owner.get((blk, slot))
            want_k = x[t, 0] if t is not None else np.full(D, 0x1234, np.uint16)
            want_v = y[t, 0] if t is not None else np.full(D, 0x4321, np.uint16)
            assert np.array_equal(kc[blk, 0, slot], want_k), (blk, slot)
            assert np.array_equal(vc[blk, 0, slot], want_v), (blk, slot)
    for gg in g["gathers"]:
        rows = gg.get("out_rows", len(gg["rows"]))
        ko = np.full((rows, H, D), 0xFFFF, np.uint16)
        vo = np.full((rows, H, D), 0xFFFF, np.uint16)
        orc.gather_bf16(kc, vc, g["block_table"], gg["context_lengths"], gg.get("offsets"), ko, vo)
        for r, tag in enumerate(gg["rows"]):
            if tag == "F":
                wk = wv = np.full(D, 0xFFFF, np.uint16)
            elif tag == "S":
                wk, wv = np.full(D, 0x1234, np.uint16), np.full(D, 0x4321, np.uint16)
            else:
                wk, wv = x[int(tag), 0], y[int(tag), 0]
            assert np.array_equal(ko[r, 0], wk) and np.array_equal(vo[r, 0], wv), (r, tag)


def pin_bf16_bruteforce(orc):
    """Random tiny problems against a dict model of logical -> physical rows."""
    rng = np.random.default_rng(777)
    for it in range(16):
        B = int(rng.integers(1, 5)); H = int(rng.integers(1, 3)); D = 16
        bs = int(rng.choice([1, 2, 4, 16])); MB = int(rng.integers(1, 5))
        NB = B * MB + int(rng.integers(0, 3)); cap = MB * bs
        ctx = rng.integers(0, cap + 1, size=B)
        q = np.array([rng.integers(0, cap - c + 1) for c in ctx])
        bt = rng.permutation(NB).astype(np.int32)[:B * MB].reshape(B, MB).copy()
        N = int(q.sum())
        x = rng.integers(0, 1 << 16, size=(N, H, D)).astype(np.uint16)
        y = rng.integers(0, 1 << 16, size=(N, H, D)).astype(np.uint16)
        kc = rng.integers(0, 1 << 16, size=(NB, H, bs, D)).astype(np.uint16)
        vc = rng.integers(0, 1 << 16, size=(NB, H, bs, D)).astype(np.uint16)
        kc0, vc0 = kc.copy(), vc.copy()
        cu = np.concatenate([[0], np.cumsum(q)]).astype(np.int32)
        orc.store_bf16(x, y, kc, vc, bt, cu, ctx.astype(np.int32))
        logical = {}
        tok = 0
        for b in range(B):
            for i in range(int(q[b])):
                logical[(b, int(ctx[b]) + i)] = tok
                tok += 1
        phys = {(int(bt[b][p // bs]), p % bs): t for (b, p), t in logical.items()}
        for blk in range(NB):
            for slot in range(bs):
                t = phys.get((blk, slot))
                assert np.array_equal(kc[blk, :, slot], kc0[blk, :, slot] if t is None else x[t])
                assert np.array_equal(vc[blk, :, slot], vc0[blk, :, slot] if t is None else y[t])
        lens = (ctx + q).astype(np.int32)
        ko, vo = orc.gather_bf16(kc, vc, bt, lens)
        row = 0
        for b in range(B):
            for p in range(int(lens[b])):
                blk, slot = int(bt[b][p // bs]), p % bs
                assert np.array_equal(ko[row], kc[blk, :, slot]) and np.array_equal(vo[row], vc[blk, :, slot])
                row += 1


# ---- paged decode attention over the int8 cache ------------------------------

def _attention_case(rng, B=3, H=2, G=2, D=16, bs=4, MB=5, mode=0, lens=None):
    NB = B * MB + 2
    kc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(NB, H, bs, D)).astype(np.int8)
    if mode == 0:
        ks = rng.uniform(0.01, 0.1, size=(NB, H, bs)).astype(np.float32)
        vs = rng.uniform(0.01, 0.1, size=(NB, H, bs)).astype(np.float32)
    elif mode == 1:
        ks = rng.uniform(0.005, 0.05, size=(H, D)).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, size=(H, D)).astype(np.float32)
    else:
        ks = rng.uniform(0.005, 0.05, size=(NB, H)).astype(np.float32)
        vs = rng.uniform(0.005, 0.05, size=(NB, H)).astype(np.float32)
    bt = rng.permutation(NB).astype(np.int32)[:B * MB].reshape(B, MB).copy()
    if lens is None:
        lens = rng.integers(0, MB * bs + 1, size=B)
    lens = np.asarray(lens, np.int32)
    q = _random_bf16_rows(rng, B, H * G, D)
    return q, kc, vc, ks, vs, bt, lens


def _attention_reference(orc, mode, q, kc, vc, ks, vs, bt, lens, scale):
    """The same attention from the gathered bf16 rows, with numpy/scipy in fp64."""
    from scipy.special import softmax
    B, HQ, D = q.shape
    H = kc.shape[1]
    G = HQ // H
    ko, vo = orc.dequant_gather(mode, kc, vc, ks, vs, bt, lens)
    kf, vf = _bits_to_f32(ko).astype(np.float64), _bits_to_f32(vo).astype(np.float64)
    qf = _bits_to_f32(q).astype(np.float64)
    off = np.concatenate([[0], np.cumsum(lens.astype(np.int64))])
    out = np.zeros((B, HQ, D))
    for b in range(B):
        if lens[b] == 0:
            continue
        kb = np.repeat(kf[off[b]:off[b + 1]], G, axis=1)  # [L][HQ][D]: query head j -> kv head j // G
        vb = np.repeat(vf[off[b]:off[b + 1]], G, axis=1)
        w = softmax(scale * np.einsum("jd,ljd->jl", qf[b], kb), axis=1)
        out[b] = np.einsum("jl,ljd->jd", w, vb)
    return out, vf, off


def pin_attention_against_library(orc):
    """Against an independent fp64 formulation on the gathered rows, for every
    scale mode, grouped heads, empty contexts and large scores."""
    rng = np.random.default_rng(61)
    for mode in (0, 1, 2):
        for scale in (0.25, 40.0):
            args = _attention_case(rng, mode=mode, lens=[0, 7, 20])
            got = orc.paged_decode_attention(mode, *args, scale)
            want, _, _ = _attention_reference(orc, mode, *args, scale)
            assert np.all(np.isfinite(got))
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (mode, scale)
            assert not got[0].any()  # empty context -> 0


def pin_attention_closed_forms(orc):
    """One position: the output is that position's V row.  Equal scores: the
    output is the mean of the V rows."""
    rng = np.random.default_rng(62)
    q, kc, vc, ks, vs, bt, lens = _attention_case(rng, B=2, G=4, lens=[1, 9])
    # sequence 1: every K code of kv head 0 equal, and one scale per position
    # that is the same, so that all its scores are equal
    for j in range(bt.shape[1]):
        kc[bt[1, j], 0] = 5
        ks[bt[1, j], 0] = np.float32(0.03)
    out = orc.paged_decode_attention(0, q, kc, vc, ks, vs, bt, lens, 0.7)
    _, vf, off = _attention_reference(orc, 0, q, kc, vc, ks, vs, bt, lens, 0.7)
    for j in range(q.shape[1]):
        h = j // 4
        assert np.array_equal(out[0, j], vf[off[0], h])        # exact: weight 1
    for j in range(4):                                          # kv head 0 of sequence 1
        assert np.allclose(out[1, j], vf[off[1]:off[2], 0].mean(axis=0), rtol=1e-13, atol=1e-15)


PINS = [pin_quantize_goldens, pin_dequant_goldens, pin_placement_golden,
        pin_exact_quantize_random, pin_exact_dequant_random, pin_invariants,
        pin_identity_table, pin_cumsum, pin_placement_bruteforce, pin_bounds_errors,
        pin_bf16_placement_golden, pin_bf16_bruteforce, pin_per_block_reduces_to_per_channel,
        pin_attention_against_library, pin_attention_closed_forms]
