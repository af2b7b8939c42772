"""Pins of the CPU oracle to facts that do not come from the oracle itself: the
hand-worked examples under tests/golden, closed forms, special cases that reduce to a
textbook routine, invariants, and defining properties checked by brute force on tiny
inputs. A plausible slip anywhere in the oracle (a dropped term, a wrong sign or index,
a transposed operand, a wrong rounding mode or cast point) fails at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from conftest import bf16_bits, bits_to_f64, read_golden

import oracle
from oracle import Dims

INT32_MIN = np.iinfo(np.int32).min


# ------------------------------------------------------------------ helpers

def paged(values_btd: list, page: int, hkv: int, perm=None):
    """Lay per-sequence [Hkv][N_b][D] float32 arrays out as a paged cache
    [pages][Hkv][page][D]; returns (cache, page_table, lens). Slots past N_b are filled
    with a recognisable junk value."""
    lens = [v.shape[1] for v in values_btd]
    D = values_btd[0].shape[2]
    pages_per = [-(-n // page) for n in lens]
    total = sum(pages_per)
    order = np.arange(total) if perm is None else np.asarray(perm)
    cache = np.full((total, hkv, page, D), 1.5, dtype=np.float32)
    pt = np.full((len(lens), max(pages_per)), -1, dtype=np.int32)
    off = 0
    for b, v in enumerate(values_btd):
        for p in range(pages_per[b]):
            pg = order[off + p]
            pt[b, p] = pg
            t0, t1 = p * page, min((p + 1) * page, lens[b])
            cache[pg, :, : t1 - t0, :] = v[:, t0:t1, :]
        off += pages_per[b]
    return cache, pt, np.asarray(lens, dtype=np.int32)


def to_bf16(x):
    """Round float32 values to bf16 (nearest even) and return them as float32."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def random_case(rng, B=1, hq=4, hkv=1, D=8, lens=(200,), page=16, perm=False):
    lens = list(lens)
    ks = [to_bf16(rng.standard_normal((hkv, n, D))) for n in lens]
    vs = [to_bf16(rng.standard_normal((hkv, n, D))) for n in lens]
    total = sum(-(-n // page) for n in lens)
    order = rng.permutation(total) if perm else None
    kc, pt, ln = paged(ks, page, hkv, order)
    vc, _, _ = paged(vs, page, hkv, order)
    q = to_bf16(rng.standard_normal((B, hq, D)))
    return dict(k=kc, v=vc, pt=pt, lens=ln, q=q, ks=ks, vs=vs, page=page)


def dims_for(case, hq, hkv, D, chunk=32, block=16, k1=4, k2=4, sink=8, window=16, scale=0.0):
    return Dims(batch=len(case["lens"]), hq=hq, hkv=hkv, head_dim=D, page_size=case["page"],
                max_pages_per_seq=case["pt"].shape[1], num_pages=case["k"].shape[0],
                chunk=chunk, block=block, k1=k1, k2=k2, sink=sink, window=window,
                sm_scale=scale)


def run_all(d, case):
    kb, vb, qb = bf16_bits(case["k"]), bf16_bits(case["v"]), bf16_bits(case["q"])
    kq, sc = oracle.quantize_keys(d, kb, case["pt"], case["lens"])
    sel = oracle.select(d, qb, sc, kq, case["pt"], case["lens"], want_block_max=True)
    out, lse = oracle.attend(d, qb, kb, vb, case["pt"], case["lens"], sel["block_idx"],
                             sel["n_blocks"])
    return kq, sc, sel, out, lse


def logical_codes(kq, pt, lens, page, hkv):
    """Per sequence [Hkv][N_b][D] view of a paged code array."""
    res = []
    for b, n in enumerate(lens):
        rows = [kq[pt[b, t // page], :, t % page, :] for t in range(n)]
        res.append(np.stack(rows, axis=1))
    return res


# ------------------------------------------------------------- worked examples

def test_key_codes_worked_example():
    g = read_golden("key_codes_d4.txt")
    keys = np.array(g["keys"], dtype=np.float32)            # [t][c]
    n, D = keys.shape
    cache, pt, lens = paged([keys[None]], int(g["page_size"]), 1)
    d = Dims(1, 1, 1, D, int(g["page_size"]), pt.shape[1], cache.shape[0], 1, 1, 0, 0, 0, 0)
    kq, sc = oracle.quantize_keys(d, bf16_bits(cache), pt, lens)
    np.testing.assert_array_equal(sc[0, 0], np.array(g["scales"][0], dtype=np.float32))
    assert sc[0, 0, 2] == np.float32(8454660 * 2.0 ** -27)
    codes = logical_codes(kq, pt, lens, int(g["page_size"]), 1)[0][0]
    np.testing.assert_array_equal(codes, np.array(g["codes"], dtype=np.int8))
    # the tail slot of the page (past N) is code 0
    assert kq[0, 0, n:, :].tolist() == [[0] * D] * (int(g["page_size"]) - n)


def test_query_codes_scores_and_modules_worked_example():
    gk = read_golden("key_codes_d4.txt")
    g = read_golden("query_scores_d4.txt")
    keys = np.array(gk["keys"], dtype=np.float32)
    q = np.array(g["query"], dtype=np.float32)[None]        # [1][G][D]
    G, D = q.shape[1], q.shape[2]
    cache, pt, lens = paged([keys[None]], int(gk["page_size"]), 1)
    d = Dims(1, G, 1, D, int(gk["page_size"]), pt.shape[1], cache.shape[0],
             int(g["chunk"]), int(g["block"]), int(g["k1"]), int(g["k2"]), int(g["sink"]),
             int(g["window"]))
    kq, sc = oracle.quantize_keys(d, bf16_bits(cache), pt, lens)
    qq, sq = oracle.query_codes(d, bf16_bits(q), sc)
    assert sq[0, 0] == np.float32(g["q_scale"])
    np.testing.assert_array_equal(qq[0, 0], np.array(g["query_codes"], dtype=np.int8))
    sel = oracle.select(d, bf16_bits(q), sc, kq, pt, lens, want_block_max=True)
    assert sel["block_max"][0, 0, :3].tolist() == [int(x) for x in g["token_scores"][0]]
    assert sel["chunk_idx"][0, 0].tolist() == [int(x) for x in g["chunk_idx"]]
    assert sel["block_idx"][0, 0].tolist() == [int(x) for x in g["block_idx"]]
    assert sel["n_blocks"][0, 0] == 2 and sel["n_chunks"][0, 0] == 3


@pytest.mark.parametrize("case_no", [0, 1, 2])
def test_tie_break_worked_example(case_no):
    g = read_golden("tie_break_d4.txt")
    c = g["cases"][case_no]
    k0 = np.array(g["key_channel0"][0], dtype=np.float32)
    keys = np.zeros((k0.size, 4), dtype=np.float32)
    keys[:, 0] = k0
    cache, pt, lens = paged([keys[None]], 4, 1)
    q = np.array(g["query"], dtype=np.float32)[None]
    k1, k2 = int(c["k1"]), int(c["k2"])
    d = Dims(1, 1, 1, 4, 4, pt.shape[1], cache.shape[0], 2, 1, k1, k2, 0, 0)
    kq, sc = oracle.quantize_keys(d, bf16_bits(cache), pt, lens)
    qq, _ = oracle.query_codes(d, bf16_bits(q), sc)
    assert qq[0, 0, 0].tolist() == [127, 0, 0, 0]
    sel = oracle.select(d, bf16_bits(q), sc, kq, pt, lens, want_block_max=True)
    assert sel["block_max"][0, 0, :8].tolist() == [4064, 8128, 8128, 2032, 16129, 4064, 8128,
                                                    -8128]
    want_c = [int(x) for x in c["chunk_idx"].split(",")]
    want_b = [int(x) for x in c["block_idx"].split(",")]
    assert sel["chunk_idx"][0, 0].tolist() == want_c + [-1] * (k1 - len(want_c))
    assert sel["block_idx"][0, 0].tolist() == want_b + [-1] * (k2 - len(want_b))


def test_attention_two_tokens_worked_example():
    g = read_golden("attention_two_tokens.txt")
    k = np.array([[0.0, 1.0], [1.0, 0.0]], dtype=np.float32)
    v = np.array([[1.0, 0.0], [0.0, 1.0]], dtype=np.float32)
    kc, pt, lens = paged([k[None]], 16, 1)
    vc, _, _ = paged([v[None]], 16, 1)
    q = np.array([[[1.0, 0.0]]], dtype=np.float32)
    d = Dims(1, 1, 1, 2, 16, 1, 1, 16, 16, 0, 0, 0, 0, sm_scale=1.0)
    out, lse = oracle.dense(d, bf16_bits(q), bf16_bits(kc), bf16_bits(vc), pt, lens)
    np.testing.assert_allclose(out[0, 0], g["out"], rtol=0, atol=1e-15)
    assert abs(lse[0, 0] - g["lse"]) < 1e-14
    # sink = window = 0 and nothing selected leaves an empty set for the sparse form...
    out2, _ = oracle.attend(d, bf16_bits(q), bf16_bits(kc), bf16_bits(vc), pt, lens,
                            np.zeros((1, 1, 0), np.int32), np.zeros((1, 1), np.int32))
    # ...and with sink 2 both tokens are attended again
    d2 = Dims(1, 1, 1, 2, 16, 1, 1, 16, 16, 0, 0, 2, 0, sm_scale=1.0)
    out3, lse3 = oracle.attend(d2, bf16_bits(q), bf16_bits(kc), bf16_bits(vc), pt, lens,
                               np.zeros((1, 1, 0), np.int32), np.zeros((1, 1), np.int32))
    np.testing.assert_allclose(out3[0, 0], g["out"], atol=1e-15)
    assert abs(lse3[0, 0] - g["lse"]) < 1e-14


# ------------------------------------------------------------ quantisation

def test_key_code_error_bound_and_extremes():
    rng = np.random.default_rng(1)
    case = random_case(rng, B=2, hq=4, hkv=2, D=16, lens=(97, 300), page=16, perm=True)
    for b in range(2):
        case["ks"][b][:, :, 3] = 0.0                         # a zero channel
        case["ks"][b][:, :, 5] *= 8.0                         # an outlier channel
    kc, pt, lens = paged(case["ks"], 16, 2, None)
    d = Dims(2, 4, 2, 16, 16, pt.shape[1], kc.shape[0], 32, 16, 2, 2, 8, 16)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, lens)
    codes = logical_codes(kq, pt, lens, 16, 2)
    for b in range(2):
        k = case["ks"][b].astype(np.float64)                 # [Hkv][N][D]
        s = sc[b].astype(np.float64)[:, None, :]
        err = np.abs(codes[b] * s - k)
        # rint of the fp32 quotient: at most half a unit plus the quotient's own rounding
        # (half an ulp of a value below 128, 2^-18)
        assert np.all(err <= s * (0.5 + 2.0 ** -17))
        amax = np.abs(k).max(axis=1)
        assert np.all(sc[b][amax > 0] > 0) and np.all(sc[b][amax == 0] == 0)
        # the element of largest magnitude of every nonzero channel codes to +-127
        top = np.abs(codes[b]).max(axis=1)
        assert np.all(top[amax > 0] == 127) and np.all(top[amax == 0] == 0)
        # codes carry the sign of the key
        assert np.all(np.sign(codes[b]) * np.sign(k) >= 0)
        # scale is the fp32 quotient amax / 127
        np.testing.assert_array_equal(sc[b], (amax / 127.0).astype(np.float32))


def test_four_bit_key_codes_worked_example():
    """The 4-bit key format by hand: one channel holding 1.75, -0.875, 0.625, 0.25, 0 (all
    exact in bf16): amax 1.75, s = f32(1.75 / 7) = 0.25 exactly; k / s = 7, -3.5, 2.5, 1, 0
    -> codes 7, -4, 2, 1, 0 (halves to even); the other channels are zero (scale 0)."""
    vals = [1.75, -0.875, 0.625, 0.25, 0.0]
    D = 8
    k = np.zeros((1, len(vals), D), dtype=np.float32)
    k[0, :, 3] = vals
    kc, pt, ln = paged([k], 16, 1)
    d = Dims(batch=1, hq=1, hkv=1, head_dim=D, page_size=16, max_pages_per_seq=pt.shape[1],
             num_pages=kc.shape[0], chunk=16, block=16, k1=1, k2=1, sink=0, window=0,
             key_bits=4)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    assert sc[0, 0, 3] == np.float32(0.25) and (np.delete(sc[0, 0], 3) == 0).all()
    assert kq[0, 0, :5, 3].tolist() == [7, -4, 2, 1, 0]
    assert (np.delete(kq[0, 0, :5], 3, axis=1) == 0).all()


@pytest.mark.parametrize("seed", range(3))
def test_four_bit_key_codes_bound_and_append(seed):
    """4-bit codes lie in [-7, 7], reach +-7 at the channel maximum, reconstruct within half a
    step (the fp32 quotient's own rounding aside), and the append of a token with the stored
    scales saturates at +-7."""
    rng = np.random.default_rng(60 + seed)
    case = random_case(rng, B=1, hq=4, hkv=2, D=16, lens=(150,))
    d = dims_for(case, 4, 2, 16)
    d.key_bits = 4
    kb = bf16_bits(case["k"])
    kq, sc = oracle.quantize_keys(d, kb, case["pt"], case["lens"])
    codes = logical_codes(kq, case["pt"], case["lens"], 16, 2)[0]       # [Hkv][N][D]
    k = case["ks"][0]
    assert codes.min() >= -7 and codes.max() <= 7
    for h in range(2):
        s = sc[0, h].astype(np.float64)
        err = np.abs(codes[h] * s[None, :] - k[h])
        assert (err <= s[None, :] * (0.5 + 2.0 ** -17)).all()
        amax_t = np.abs(k[h]).argmax(axis=0)
        assert (np.abs(codes[h][amax_t, np.arange(16)]) == 7).all()
    # append: a token far beyond the stored scales saturates
    kc2 = case["k"].copy()
    n = int(case["lens"][0])
    kc2[case["pt"][0, (n - 1) // 16], :, (n - 1) % 16, :] = 100.0
    kq2 = oracle.quantize_append(d, bf16_bits(kc2), case["pt"], case["lens"], -1, sc, kq)
    last = logical_codes(kq2, case["pt"], case["lens"], 16, 2)[0][:, n - 1, :]
    assert ((last == 7) | (sc[0] == 0)).all()


@pytest.mark.parametrize("m", [-3, 2])
def test_power_of_two_rescale_invariance(m):
    rng = np.random.default_rng(2)
    case = random_case(rng, B=1, hq=4, hkv=1, D=16, lens=(400,), page=16)
    d = dims_for(case, 4, 1, 16, chunk=32, block=16, k1=4, k2=3, sink=8, window=16)
    kq, sc, sel, out, _ = run_all(d, case)
    case2 = dict(case)
    case2["k"] = case["k"] * np.float32(2.0 ** m)
    case2["q"] = case["q"] * np.float32(2.0 ** -m)
    kq2, sc2, sel2, out2, _ = run_all(d, case2)
    np.testing.assert_array_equal(kq2, kq)
    np.testing.assert_array_equal(sc2, sc * np.float32(2.0 ** m))
    for key in ("chunk_idx", "block_idx", "block_max"):
        np.testing.assert_array_equal(sel2[key], sel[key])
    np.testing.assert_allclose(out2, out, atol=1e-12)


def test_page_permutation_invariance():
    rng = np.random.default_rng(3)
    base = random_case(rng, B=3, hq=8, hkv=2, D=16, lens=(150, 33, 260), page=16)
    total = base["k"].shape[0]
    perm = rng.permutation(total)
    kc, pt, lens = paged(base["ks"], 16, 2, perm)
    vc, _, _ = paged(base["vs"], 16, 2, perm)
    other = dict(base, k=kc, v=vc, pt=pt)
    d = dims_for(base, 8, 2, 16, chunk=32, block=16, k1=3, k2=3, sink=8, window=16)
    kq, sc, sel, out, lse = run_all(d, base)
    kq2, sc2, sel2, out2, lse2 = run_all(d, other)
    for a, b in zip(logical_codes(kq, base["pt"], lens, 16, 2), logical_codes(kq2, pt, lens, 16, 2)):
        np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(sc, sc2)
    for key in ("chunk_idx", "block_idx", "n_blocks", "block_max"):
        np.testing.assert_array_equal(sel[key], sel2[key])
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_append_reuses_stored_scales_and_saturates():
    rng = np.random.default_rng(4)
    case = random_case(rng, B=2, hq=4, hkv=2, D=16, lens=(70, 129), page=16)
    d = dims_for(case, 4, 2, 16)
    kb = bf16_bits(case["k"])
    kq, sc = oracle.quantize_keys(d, kb, case["pt"], case["lens"])
    wiped = kq.copy()
    for b, n in enumerate(case["lens"]):
        wiped[case["pt"][b, (n - 1) // 16], :, (n - 1) % 16, :] = 0
    again = oracle.quantize_append(d, kb, case["pt"], case["lens"], -1, sc, wiped)
    np.testing.assert_array_equal(again, kq)
    # a new last token beyond the stored range saturates at +-127
    big = case["k"].copy()
    for b, n in enumerate(case["lens"]):
        big[case["pt"][b, (n - 1) // 16], :, (n - 1) % 16, :] = 64.0
        big[case["pt"][b, (n - 1) // 16], :, (n - 1) % 16, 0] = -64.0
    sat = oracle.quantize_append(d, bf16_bits(big), case["pt"], case["lens"], -1, sc, kq)
    for b, n in enumerate(case["lens"]):
        row = sat[case["pt"][b, (n - 1) // 16], :, (n - 1) % 16, :]
        assert np.all(row[:, 1:] == 127) and np.all(row[:, 0] == -127)


def test_query_codes_bound_and_zero():
    rng = np.random.default_rng(5)
    case = random_case(rng, B=2, hq=8, hkv=2, D=16, lens=(50, 80), page=16)
    d = dims_for(case, 8, 2, 16)
    kq, sc = oracle.quantize_keys(d, bf16_bits(case["k"]), case["pt"], case["lens"])
    qq, sq = oracle.query_codes(d, bf16_bits(case["q"]), sc)
    G = 4
    for b in range(2):
        for h in range(2):
            qf = (case["q"][b, h * G:(h + 1) * G].astype(np.float64) * sc[b, h]).astype(np.float32)
            assert np.abs(qq[b, h]).max() == 127
            err = np.abs(qq[b, h] * np.float64(sq[b, h]) - qf)
            assert np.all(err <= sq[b, h] * (0.5 + 2.0 ** -17))
    qz, sz = oracle.query_codes(d, bf16_bits(np.zeros_like(case["q"])), sc)
    assert not qz.any() and not sz.any()


# ---------------------------------------------------------------- selection

def _block_max_by_definition(qq, codes, n, sink, window, block):
    """Block maxima written from the definition: every candidate token's score is the
    largest of the group's integer dot products."""
    lo, hi = sink, n - window
    out = {}
    for t in range(lo, hi):
        g = max(int(np.dot(qq[j].astype(np.int64), codes[t].astype(np.int64)))
                for j in range(qq.shape[0]))
        out[t // block] = max(out.get(t // block, g), g)
    return out


def _beats(a_score, a_idx, b_score, b_idx):
    return a_score > b_score or (a_score == b_score and a_idx < b_idx)


@pytest.mark.parametrize("seed", range(6))
def test_modules_defining_property_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    D, hkv, G = 8, 2, 2
    lens = tuple(int(x) for x in rng.integers(1, 520, size=2))
    case = random_case(rng, B=2, hq=hkv * G, hkv=hkv, D=D, lens=lens, page=16, perm=True)
    block = int(rng.choice([16, 32]))
    chunk = block * int(rng.choice([1, 2, 4]))
    k1, k2 = int(rng.integers(0, 9)), int(rng.integers(0, 12))
    sink, window = int(rng.integers(0, 40)), int(rng.integers(0, 60))
    # integer-valued keys make ties frequent
    for b in range(2):
        case["ks"][b] = np.round(case["ks"][b] * 2) / 2
    kc, pt, ln = paged(case["ks"], 16, hkv, None)
    case.update(k=kc, pt=pt)
    d = dims_for(case, hkv * G, hkv, D, chunk=chunk, block=block, k1=k1, k2=k2, sink=sink,
                 window=window)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    qq, _ = oracle.query_codes(d, bf16_bits(case["q"]), sc)
    sel = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln, want_block_max=True)
    codes = logical_codes(kq, pt, ln, 16, hkv)
    per = chunk // block
    for b in range(2):
        for h in range(hkv):
            n = int(ln[b])
            bm = _block_max_by_definition(qq[b, h], codes[b][h], n, sink, window, block)
            got = sel["block_max"][b, h]
            for k in range(got.size):
                assert got[k] == bm.get(k, INT32_MIN)
            cm = {}
            for k, s in bm.items():
                cm[k // per] = max(cm.get(k // per, s), s)
            kept_c = [c for c in sel["chunk_idx"][b, h] if c >= 0]
            assert kept_c == sorted(kept_c) and len(kept_c) == min(k1, len(cm))
            assert sel["n_chunks"][b, h] == len(kept_c)
            for c in kept_c:
                for c2 in cm:
                    if c2 not in kept_c:
                        assert _beats(cm[c], c, cm[c2], c2)
            cand = [k for k in bm if k // per in kept_c]
            kept_b = [k for k in sel["block_idx"][b, h] if k >= 0]
            assert kept_b == sorted(kept_b) and len(kept_b) == min(k2, len(cand))
            assert sel["n_blocks"][b, h] == len(kept_b)
            for k in kept_b:
                assert k in cand
                for k2_ in cand:
                    if k2_ not in kept_b:
                        assert _beats(bm[k], k, bm[k2_], k2_)
            if k1 >= k2:
                # closed form: the two stages equal the single-stage top-K2 of all blocks
                ranked = sorted(bm, key=lambda k: (-bm[k], k))[:k2]
                assert sorted(ranked) == kept_b


@pytest.mark.parametrize("seed", range(8))
def test_module1_keeping_k2_chunks_keeps_the_same_blocks(seed):
    """With K1 >= K2, module 1 keeping only the top K2 chunks leaves module 2's kept blocks
    unchanged: every chunk ranked above a kept block's chunk holds a block ranked above that
    block. The whole decode step relies on this (it outputs no chunk ids)."""
    rng = np.random.default_rng(700 + seed)
    D, hkv, G = 8, 2, 2
    lens = tuple(int(x) for x in rng.integers(64, 900, size=2))
    case = random_case(rng, B=2, hq=hkv * G, hkv=hkv, D=D, lens=lens, page=16, perm=True)
    for b in range(2):
        case["ks"][b] = np.round(case["ks"][b] * 2) / 2  # frequent ties
    kc, pt, ln = paged(case["ks"], 16, hkv, None)
    case.update(k=kc, pt=pt)
    k2 = int(rng.integers(1, 10))
    k1 = k2 + int(rng.integers(0, 8))
    d = dims_for(case, hkv * G, hkv, D, chunk=64, block=16, k1=k1, k2=k2,
                 sink=int(rng.integers(0, 40)), window=int(rng.integers(1, 60)))
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    full = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln)
    d.k1 = k2
    short = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln)
    np.testing.assert_array_equal(full["block_idx"], short["block_idx"])
    np.testing.assert_array_equal(full["n_blocks"], short["n_blocks"])
    # and every kept block reaches T1, the K2-th largest chunk maximum (the top K2 chunks each
    # hold a block equal to their maximum), the bound the whole step's selection starts from
    sel = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln, want_block_max=True)
    for b in range(2):
        for h in range(hkv):
            bm = sel["block_max"][b, h].astype(np.int64)
            nblk = bm.size
            cm = np.full((nblk + 3) // 4, INT32_MIN, dtype=np.int64)
            for k in range(nblk):
                cm[k // 4] = max(cm[k // 4], bm[k])
            valid = np.sort(cm[cm != INT32_MIN])[::-1]
            if valid.size < k2:
                continue
            t1 = valid[k2 - 1]
            kept = [k for k in sel["block_idx"][b, h] if k >= 0]
            assert len(kept) == k2 and all(bm[k] >= t1 for k in kept)
            assert (bm >= t1).sum() >= k2


@pytest.mark.parametrize("seed", range(6))
def test_three_stacked_modules_defining_property_brute_force(seed):
    """A first module on coarse chunks (chunk0 tokens) keeps the top K0; module 1 ranks only
    the fine chunks inside them; module 2 as before. Each stage is checked by brute force
    against its defining property, and with K0 >= K1 the three stages equal the two."""
    rng = np.random.default_rng(300 + seed)
    D, hkv, G = 8, 2, 2
    lens = tuple(int(x) for x in rng.integers(100, 900, size=2))
    case = random_case(rng, B=2, hq=hkv * G, hkv=hkv, D=D, lens=lens, page=16, perm=True)
    for b in range(2):
        case["ks"][b] = np.round(case["ks"][b] * 2) / 2  # frequent ties
    kc, pt, ln = paged(case["ks"], 16, hkv, None)
    case.update(k=kc, pt=pt)
    block, chunk = 16, 32
    chunk0 = chunk * int(rng.choice([2, 4]))
    k0, k1, k2 = int(rng.integers(1, 6)), int(rng.integers(1, 12)), int(rng.integers(0, 14))
    sink, window = int(rng.integers(0, 40)), int(rng.integers(0, 60))
    d = dims_for(case, hkv * G, hkv, D, chunk=chunk, block=block, k1=k1, k2=k2, sink=sink,
                 window=window)
    d.chunk0, d.k0 = chunk0, k0
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    qq, _ = oracle.query_codes(d, bf16_bits(case["q"]), sc)
    sel = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln)
    codes = logical_codes(kq, pt, ln, 16, hkv)
    per, per0 = chunk // block, chunk0 // block
    for b in range(2):
        for h in range(hkv):
            bm = _block_max_by_definition(qq[b, h], codes[b][h], int(ln[b]), sink, window, block)
            cm0, cm = {}, {}
            for k, s_ in bm.items():
                cm0[k // per0] = max(cm0.get(k // per0, s_), s_)
                cm[k // per] = max(cm.get(k // per, s_), s_)
            kept0 = sorted(cm0, key=lambda c: (-cm0[c], c))[:k0]
            for c in kept0:
                for c2 in cm0:
                    if c2 not in kept0:
                        assert _beats(cm0[c], c, cm0[c2], c2)
            cand1 = [c for c in cm if c * chunk // chunk0 in kept0]
            kept_c = [c for c in sel["chunk_idx"][b, h] if c >= 0]
            assert kept_c == sorted(kept_c) and len(kept_c) == min(k1, len(cand1))
            for c in kept_c:
                assert c in cand1
                for c2 in cand1:
                    if c2 not in kept_c:
                        assert _beats(cm[c], c, cm[c2], c2)
            cand2 = [k for k in bm if k // per in kept_c]
            kept_b = [k for k in sel["block_idx"][b, h] if k >= 0]
            assert kept_b == sorted(kept_b) and len(kept_b) == min(k2, len(cand2))
            for k in kept_b:
                assert k in cand2
                for k_ in cand2:
                    if k_ not in kept_b:
                        assert _beats(bm[k], k, bm[k_], k_)
    # closed form: a coarse chunk holding a top-K1 fine chunk is itself in the top K1 coarse
    # chunks, so with K0 >= K1 module 0 removes nothing that module 1 would keep
    d.k0 = max(k1, 1)
    three = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln)
    d.k0 = 0
    two = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln)
    for key in ("chunk_idx", "n_chunks", "block_idx", "n_blocks"):
        np.testing.assert_array_equal(three[key], two[key])


@pytest.mark.parametrize("seed", range(5))
def test_per_head_selection_defining_property_brute_force(seed):
    """Per-head selection (InfiniteHiP article, stacked modules: every head prunes on its
    own): each query head ranks its own integer dot products, with the group's shared
    query codes and no max over the group. Checked by brute force row by row, and by the
    closed form that a kv head's shared block maximum is the max of its heads' maxima."""
    rng = np.random.default_rng(500 + seed)
    D, hkv, G = 8, 2, 2 + 2 * (seed % 2)
    lens = tuple(int(x) for x in rng.integers(60, 600, size=2))
    case = random_case(rng, B=2, hq=hkv * G, hkv=hkv, D=D, lens=lens, page=16, perm=True)
    for b in range(2):
        case["ks"][b] = np.round(case["ks"][b] * 2) / 2  # frequent ties
    kc, pt, ln = paged(case["ks"], 16, hkv, None)
    case.update(k=kc, pt=pt)
    k1, k2 = int(rng.integers(1, 9)), int(rng.integers(0, 12))
    sink, window = int(rng.integers(0, 40)), int(rng.integers(0, 60))
    d = dims_for(case, hkv * G, hkv, D, chunk=32, block=16, k1=k1, k2=k2, sink=sink,
                 window=window)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    qq, _ = oracle.query_codes(d, bf16_bits(case["q"]), sc)
    shared = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln, want_block_max=True)
    d.per_head = 1
    ph = oracle.select(d, bf16_bits(case["q"]), sc, kq, pt, ln, want_block_max=True)
    assert ph["block_idx"].shape == (2, hkv * G, k2)
    codes = logical_codes(kq, pt, ln, 16, hkv)
    for b in range(2):
        for h in range(hkv):
            for j in range(G):
                row = h * G + j
                bm = _block_max_by_definition(qq[b, h, j:j + 1], codes[b][h], int(ln[b]), sink,
                                              window, 16)
                got = ph["block_max"][b, row]
                for k in range(got.size):
                    assert got[k] == bm.get(k, INT32_MIN)
                cm = {}
                for k, s_ in bm.items():
                    cm[k // 2] = max(cm.get(k // 2, s_), s_)
                kept_c = [c for c in ph["chunk_idx"][b, row] if c >= 0]
                assert kept_c == sorted(kept_c) and len(kept_c) == min(k1, len(cm))
                for c in kept_c:
                    for c2 in cm:
                        if c2 not in kept_c:
                            assert _beats(cm[c], c, cm[c2], c2)
                cand = [k for k in bm if k // 2 in kept_c]
                kept_b = [k for k in ph["block_idx"][b, row] if k >= 0]
                assert kept_b == sorted(kept_b) and len(kept_b) == min(k2, len(cand))
                assert ph["n_blocks"][b, row] == len(kept_b)
                for k in kept_b:
                    for k_ in cand:
                        if k_ not in kept_b:
                            assert _beats(bm[k], k, bm[k_], k_)
            # max over the group commutes with the per-block max
            np.testing.assert_array_equal(
                shared["block_max"][b, h], ph["block_max"][b, h * G:(h + 1) * G].max(axis=0))


def test_per_head_selection_special_cases():
    """One query head per kv head: per-head selection is the shared one. Identical query
    heads in a group: every head's row is the group's shared selection."""
    rng = np.random.default_rng(77)
    case = random_case(rng, B=2, hq=2, hkv=2, D=8, lens=(300, 410), page=16)
    d = dims_for(case, 2, 2, 8, k1=5, k2=7, sink=16, window=32)
    kq, sc = oracle.quantize_keys(d, bf16_bits(case["k"]), case["pt"], case["lens"])
    a = oracle.select(d, bf16_bits(case["q"]), sc, kq, case["pt"], case["lens"])
    d.per_head = 1
    b_ = oracle.select(d, bf16_bits(case["q"]), sc, kq, case["pt"], case["lens"])
    for key in a:
        np.testing.assert_array_equal(a[key], b_[key])
    case = random_case(rng, B=1, hq=8, hkv=2, D=8, lens=(500,), page=16)
    case["q"][0, 4:8] = case["q"][0, 4]
    case["q"][0, 0:4] = case["q"][0, 1]
    d = dims_for(case, 8, 2, 8, k1=6, k2=9, sink=16, window=32)
    kq, sc = oracle.quantize_keys(d, bf16_bits(case["k"]), case["pt"], case["lens"])
    shared = oracle.select(d, bf16_bits(case["q"]), sc, kq, case["pt"], case["lens"])
    d.per_head = 1
    ph = oracle.select(d, bf16_bits(case["q"]), sc, kq, case["pt"], case["lens"])
    for key in shared:
        for j in range(8):
            np.testing.assert_array_equal(ph[key][0, j], shared[key][0, j // 4])


def test_per_head_attention_reads_each_heads_own_row():
    """With per-head selection query head j attends to the blocks of row j: the same as a
    shared-selection attention whose kv head row holds head j's list."""
    rng = np.random.default_rng(78)
    case = random_case(rng, B=1, hq=4, hkv=2, D=8, lens=(400,), page=16)
    d = dims_for(case, 4, 2, 8, k1=8, k2=6, sink=16, window=32)
    kb, vb, qb = bf16_bits(case["k"]), bf16_bits(case["v"]), bf16_bits(case["q"])
    n_cand = (400 - 32) // 16
    lists = np.stack([np.sort(rng.choice(np.arange(1, n_cand), size=6, replace=False))
                      for _ in range(4)]).astype(np.int32)[None]
    counts = np.array([[6, 5, 3, 0]], dtype=np.int32)
    d.per_head = 1
    out_ph, lse_ph = oracle.attend(d, qb, kb, vb, case["pt"], case["lens"], lists, counts)
    d.per_head = 0
    for j in range(4):
        h = j // 2
        row = np.full((1, 2, 6), -1, dtype=np.int32)
        row[0, h] = lists[0, j]
        cnt = np.zeros((1, 2), dtype=np.int32)
        cnt[0, h] = counts[0, j]
        out_s, lse_s = oracle.attend(d, qb, kb, vb, case["pt"], case["lens"], row, cnt)
        np.testing.assert_array_equal(out_ph[0, j], out_s[0, j])
        assert lse_ph[0, j] == lse_s[0, j]


# ------------------------------------------------------------------ FP8 keys

def _ordered_to_float(keys):
    """Inverse of the oracle's ordered integer of an fp32 score."""
    k = np.asarray(keys, dtype=np.int64)
    bits = np.where(k >= 0, k, k ^ 0x7FFFFFFF).astype(np.int64) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_fp8_key_codes_match_the_library_conversion():
    """FP8 keys ("KV Cache 与长上下文推理", section "KV Cache 量化": FP8 KV caches): scale
    f32(amax / 448), code = E4M3 of f32(k / s), rounded to nearest with ties to even. Pinned
    against PyTorch's float8_e4m3fn conversion (every |x| here is at most 448, where the
    two agree), and the decoded codes against the half-step bound."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    case = random_case(rng, B=2, hq=4, hkv=2, D=16, lens=(70, 45), page=16, perm=True)
    for b in range(2):  # wide dynamic range: tiny, subnormal-range and large values
        case["ks"][b] = to_bf16(case["ks"][b] * np.exp2(rng.integers(-12, 6, size=(2, 1, 16))))
    kc, pt, ln = paged(case["ks"], 16, 2, None)
    d = dims_for(dict(case, k=kc, pt=pt), 4, 2, 16)
    d.key_fp8 = 1
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    for b in range(2):
        for h in range(2):
            n = int(ln[b])
            keys = case["ks"][b][h].astype(np.float32)                   # [n][D]
            amax = np.abs(keys).max(axis=0)
            s = (amax.astype(np.float64) / 448.0).astype(np.float32)
            np.testing.assert_array_equal(sc[b, h], s)
            x = (keys / s).astype(np.float32)                             # f32 quotient
            assert np.abs(x).max() <= 448.0 + 1e-3
            want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            got = logical_codes(kq, pt, ln, 16, 2)[b][h].view(np.uint8)[:n]
            np.testing.assert_array_equal(got, want)
            dec = torch.from_numpy(got.copy()).view(torch.float8_e4m3fn).float().numpy()
            # half a step of the E4M3 grid: 2^-4 relative for normals, 2^-10 absolute below
            bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10)
            assert np.all(np.abs(dec - x) <= bound)


def test_fp8_worked_examples_and_saturating_append():
    """Hand-worked E4M3 codes with s = 1 (amax 448): 1.0625 ties to 1.0 (even mantissa),
    1.1875 ties to 1.25, 3 x 2^-10 ties to 2^-8 and 2^-10 to 0 on the subnormal grid, -0 keeps
    its sign; an appended key beyond the stored range saturates at +-448."""
    d = Dims(batch=1, hq=1, hkv=1, head_dim=4, page_size=16, max_pages_per_seq=1,
             num_pages=1, chunk=16, block=16, k1=1, k2=1, sink=0, window=0, key_fp8=1)
    k = np.zeros((1, 1, 16, 4), np.float32)
    k[0, 0, :8, 0] = [448.0, 1.0625, 1.1875, 3 * 2.0 ** -10, 2.0 ** -10, -1.0625, -0.0, 7.5]
    pt, ln = np.zeros((1, 1), np.int32), np.array([8], np.int32)
    kq, sc = oracle.quantize_keys(d, bf16_bits(k), pt, ln)
    assert sc[0, 0, 0] == 1.0 and sc[0, 0, 1] == 0.0
    # codes: sign | exponent field << 3 | mantissa
    assert kq[0, 0, :8, 0].view(np.uint8).tolist() == [0x7E, 0x38, 0x3A, 0x02, 0x00, 0xB8, 0x80,
                                                      0x4F]
    assert (kq[0, 0, :8, 1:] == 0).all() and (kq[0, 0, 8:] == 0).all()
    k[0, 0, 8, 0] = 1000.0
    k[0, 0, 8, 1] = -600.0
    ln2 = np.array([9], np.int32)
    kq2 = oracle.quantize_append(d, bf16_bits(k), pt, ln2, -1, sc, kq)
    assert kq2[0, 0, 8, 0].view(np.uint8) == 0x7E  # +448
    assert kq2[0, 0, 8, 1] == 0  # channel 1 has scale 0: code 0


@pytest.mark.parametrize("seed", range(4))
def test_fp8_scores_exact_on_representable_inputs(seed):
    """Keys that are E4M3 integers times s = 1/8 and queries that are small integers make
    every product and partial sum exact, so the scores must equal the exact rational dot
    products: block maxima (max over the group, candidate tokens only) checked against exact
    arithmetic (the exact scores of fp8_block_scores and the fp32 block_max output alike),
    and both modules against their defining property."""
    rng = np.random.default_rng(700 + seed)
    D, hkv, G = 16, 2, 2
    grid = np.array([v for v in range(1, 449) if v <= 16 or (v <= 32 and v % 2 == 0) or
                     (v <= 64 and v % 4 == 0) or (v <= 128 and v % 8 == 0) or
                     (v <= 256 and v % 16 == 0) or v % 32 == 0 and v <= 448], dtype=np.float64)
    lens = tuple(int(x) for x in rng.integers(100, 500, size=2))
    ks = []
    for n in lens:
        x = rng.choice(grid[grid <= 64], size=(hkv, n, D)) * rng.choice([-1, 1], size=(hkv, n, D))
        x[:, rng.integers(0, n), :] = 448.0  # amax 448 in every channel: s = 448/8/448 = 1/8
        ks.append((x / 8.0).astype(np.float32))
    kc, pt, ln = paged(ks, 16, hkv, None)
    qint = rng.integers(-8, 9, size=(2, hkv * G, D))
    case = dict(k=kc, pt=pt, lens=ln, page=16)
    k1, k2 = int(rng.integers(1, 8)), int(rng.integers(1, 10))
    sink, window = int(rng.integers(0, 30)), int(rng.integers(0, 50))
    d = dims_for(case, hkv * G, hkv, D, chunk=32, block=16, k1=k1, k2=k2, sink=sink,
                 window=window)
    d.key_fp8 = 1
    q = qint.astype(np.float32)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    assert np.all(sc == np.float32(1.0 / 8.0))
    sel = oracle.select(d, bf16_bits(q), sc, kq, pt, ln, want_block_max=True)
    exact, bound = oracle.fp8_block_scores(d, bf16_bits(q), sc, kq, pt, ln)
    for b in range(2):
        n = int(ln[b])
        for h in range(hkv):
            keys8 = (ks[b][h].astype(np.float64) * 8).astype(np.int64)  # exact E4M3 values
            bm = {}
            for t in range(sink, n - window):
                # q' = q / 8 exactly, key value = keys8: score = sum(q * keys8) / 8
                g = max(int(np.dot(qint[b, h * G + j], keys8[t])) for j in range(G))
                bm[t // 16] = max(bm.get(t // 16, g), g)
            got = _ordered_to_float(sel["block_max"][b, h])
            for kk in range(got.size):
                if kk in bm:
                    assert got[kk] == bm[kk] / 8.0
                    assert exact[b, h, kk] == bm[kk] / 8.0 and bound[b, h, kk] > 0
                else:
                    assert sel["block_max"][b, h, kk] == INT32_MIN
                    assert exact[b, h, kk] == -np.inf
            cm = {}
            for kk, s_ in bm.items():
                cm[kk // 2] = max(cm.get(kk // 2, s_), s_)
            kept_c = [c for c in sel["chunk_idx"][b, h] if c >= 0]
            assert len(kept_c) == min(k1, len(cm))
            for c in kept_c:
                for c2 in cm:
                    if c2 not in kept_c:
                        assert _beats(cm[c], c, cm[c2], c2)
            cand = [kk for kk in bm if kk // 2 in kept_c]
            kept_b = [kk for kk in sel["block_idx"][b, h] if kk >= 0]
            assert len(kept_b) == min(k2, len(cand))
            for kk in kept_b:
                for k_ in cand:
                    if k_ not in kept_b:
                        assert _beats(bm[kk], kk, bm[k_], k_)


def _fma32(a, b, c):
    """IEEE fp32 fused multiply-add a * b + c with one rounding, for float32 arrays: the
    product is exact in fp64, TwoSum gives the fp64 sum's exact error, and a sum that lands
    exactly halfway between two fp32 values is settled by that error's sign."""
    a64, b64, c64 = (np.asarray(x, dtype=np.float64) for x in (a, b, c))
    p = a64 * b64
    s = p + c64
    bv = s - p
    err = (p - (s - bv)) + (c64 - bv)
    r = s.astype(np.float32)
    r64 = r.astype(np.float64)
    other = np.nextafter(r, np.where(s > r64, np.float32(np.inf), np.float32(-np.inf)))
    o64 = other.astype(np.float64)
    mid = (s != r64) & (s == (r64 + o64) / 2)
    fix = mid & (err != 0) & ((err > 0) == (o64 > r64))
    return np.where(fix, other, r)


def test_fma32_emulation_worked_examples():
    """The fp32 fused multiply-add emulation: exact cases, a product below half an ulp of
    the addend that a separately rounded product would lose, and a sum that an fp64 add
    leaves exactly halfway between two fp32 values (settled by the exact remainder)."""
    f = np.float32
    assert _fma32(f(3), f(5), f(7)) == f(22)
    # 1 + 2^-24 * (1 + 2^-23): the exact sum lies just above the midpoint 1 + 2^-24
    a, b = f(2.0 ** -24), f(1 + 2.0 ** -23)
    assert _fma32(a, b, f(1.0)) == np.nextafter(f(1.0), f(2.0))
    # a product of 2^-24 exactly: a tie, to even (1.0)
    assert _fma32(f(2.0 ** -12), f(2.0 ** -12), f(1.0)) == f(1.0)
    # fp64 rounds 1 + 2^-24 + 2^-80 to the midpoint 1 + 2^-24; the remainder decides: up
    a, b = f(2.0 ** -24 * (1 + 2.0 ** -23)), f(1 + 2.0 ** -23)
    exact_above_mid = _fma32(a, b, f(1.0))
    assert exact_above_mid == np.nextafter(f(1.0), f(2.0))


def _two_modules(bm_row, k1, k2, per):
    """Both modules by their definition on one row of block scores (-inf: no candidate)."""
    cs = {}
    for k in np.nonzero(np.isfinite(bm_row))[0]:
        cs[k // per] = max(cs.get(k // per, -np.inf), bm_row[k])
    kept_c = sorted(sorted(cs, key=lambda c: (-cs[c], c))[:k1])
    cand = [k for c in kept_c for k in range(c * per, c * per + per)
            if k < bm_row.size and np.isfinite(bm_row[k])]
    return kept_c, sorted(sorted(cand, key=lambda k: (-bm_row[k], k))[:k2])


def _as_selection(d, rows):
    """[1][R][K] padded arrays of (kept chunks, kept blocks) lists, one per row."""
    R = len(rows)
    ci = np.full((1, R, d.k1), -1, np.int32)
    bi = np.full((1, R, d.k2), -1, np.int32)
    nc = np.zeros((1, R), np.int32)
    nb = np.zeros((1, R), np.int32)
    for r, (kc, kb) in enumerate(rows):
        ci[0, r, :len(kc)] = kc
        bi[0, r, :len(kb)] = kb
        nc[0, r], nb[0, r] = len(kc), len(kb)
    return ci, nc, bi, nb


@pytest.mark.parametrize("seed", range(3))
def test_fp8_exact_scores_bound_an_fp32_chain(seed):
    """FP8 scores on inputs fp32 cannot represent exactly. The oracle's exact block scores
    (fp8_block_scores) against an fp32 chain of fused multiply-adds in channel order,
    emulated here with one rounding per term: every chain block maximum lies within the
    oracle's bound, some differ from the exact score (the bound is exercised), and the
    bound equals Higham's gamma_128 (recursive summation, u = 2^-24) times the largest
    sum |q' x| of the block computed here. The validity check accepts the chain's own
    two-module selection and the oracle's, and rejects one kept block swapped for a clearly
    worse candidate, and a count one short (the weakest kept block left out)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(900 + seed)
    D, hkv, G = 128, 2, 4
    n = int(rng.integers(300, 700))
    case = random_case(rng, B=1, hq=hkv * G, hkv=hkv, D=D, lens=(n,), perm=True)
    for h in range(hkv):  # outlier channels, as in the workloads
        case["ks"][0][h][:, rng.choice(D, 4, replace=False)] *= 8
    case["k"], case["pt"], case["lens"] = paged(case["ks"], 16, hkv, rng.permutation(
        case["k"].shape[0]))
    k1, k2, sink, window, per = 6, 9, 16, 40, 4
    d = dims_for(case, hkv * G, hkv, D, chunk=64, block=16, k1=k1, k2=k2, sink=sink,
                 window=window)
    d.key_fp8 = 1
    kb, qb = bf16_bits(case["k"]), bf16_bits(case["q"])
    kq, sc = oracle.quantize_keys(d, kb, case["pt"], case["lens"])
    score, bound = oracle.fp8_block_scores(d, qb, sc, kq, case["pt"], case["lens"])
    codes = logical_codes(kq, case["pt"], case["lens"], 16, hkv)[0]  # [Hkv][n][D]
    x = torch.from_numpy(codes.view(np.uint8).copy()).view(torch.float8_e4m3fn).float().numpy()
    u = 2.0 ** -24
    gamma = 128 * u / (1 - 128 * u)
    rows = []
    for h in range(hkv):
        qf = case["q"][0, h * G:(h + 1) * G].astype(np.float32) * sc[0, h]  # fp32 products
        acc = np.zeros((G, n), np.float32)
        for c in range(D):
            acc = _fma32(np.broadcast_to(qf[:, c:c + 1], (G, n)),
                         np.broadcast_to(x[h, :, c], (G, n)), acc)
        mag = np.abs(qf.astype(np.float64)[:, None, :] * x[h].astype(np.float64)[None]).sum(-1)
        chain = np.full(d.max_blocks, -np.inf)
        want_bound = np.zeros(d.max_blocks)
        for t in range(sink, n - window):
            chain[t // 16] = max(chain[t // 16], acc[:, t].max())
            want_bound[t // 16] = max(want_bound[t // 16], gamma * mag[:, t].max())
        valid = np.isfinite(score[0, h])
        assert (np.isfinite(chain) == valid).all()
        diff = np.abs(chain[valid] - score[0, h][valid])
        assert (diff <= bound[0, h][valid]).all()
        assert (diff > 0).any()
        np.testing.assert_allclose(bound[0, h][valid], want_bound[valid], rtol=1e-12)
        rows.append(_two_modules(chain, k1, k2, per))
    lens = case["lens"]
    assert oracle.selection_within_bounds(d, lens, score, bound, *_as_selection(d, rows)) == []
    sel = oracle.select(d, qb, sc, kq, case["pt"], lens)
    assert oracle.selection_within_bounds(d, lens, score, bound, sel["chunk_idx"],
                                          sel["n_chunks"], sel["block_idx"],
                                          sel["n_blocks"]) == []
    # planted mistakes: the best kept block replaced by the worst candidate; a short count
    kc0, kb0 = rows[0]
    cand = [k for c in kc0 for k in range(c * per, c * per + per) if np.isfinite(score[0, 0, k])]
    best = max(kb0, key=lambda k: score[0, 0, k])
    worst = min(set(cand) - set(kb0), key=lambda k: score[0, 0, k])
    assert score[0, 0, best] - bound[0, 0, best] > score[0, 0, worst] + bound[0, 0, worst]
    swapped = [(kc0, sorted(set(kb0) - {best} | {worst}))] + rows[1:]
    bad = oracle.selection_within_bounds(d, lens, score, bound, *_as_selection(d, swapped))
    assert [v[2] for v in bad] == ["block order"]
    short = [(kc0, sorted(set(kb0) - {min(kb0, key=lambda k: score[0, 0, k])}))] + rows[1:]
    bad = oracle.selection_within_bounds(d, lens, score, bound, *_as_selection(d, short))
    assert [v[2] for v in bad] == ["block count"]


def test_candidate_region_masks_sink_and_window_tokens():
    """A huge key in the sink part of a block that straddles the sink boundary, and one in
    the window, must not lift any block score."""
    D, n, sink, window = 4, 64, 8, 20
    keys = np.zeros((n, D), dtype=np.float32)
    keys[3, 0] = 8.0       # sink token inside block 0
    keys[50, 0] = 8.0      # window token (window = [44, 64)) inside block 3 = [48, 64)
    keys[10, 0] = 1.0      # candidate token in block 0
    keys[40, 0] = 0.5      # candidate token in block 2
    keys[46, 0] = 0.25     # candidate token of block 2 (block 2 = [32, 48) straddles 44)
    kc, pt, ln = paged([keys[None]], 16, 1)
    q = np.array([[[1.0, 0, 0, 0]]], dtype=np.float32)
    d = Dims(1, 1, 1, D, 16, pt.shape[1], kc.shape[0], 16, 16, 4, 4, sink, window)
    kq, sc = oracle.quantize_keys(d, bf16_bits(kc), pt, ln)
    sel = oracle.select(d, bf16_bits(q), sc, kq, pt, ln, want_block_max=True)
    # s = f32(8/127): keys 1, 0.5, 0.25 code to 16, 8, 4; the query codes are (127, 0, 0, 0)
    codes = logical_codes(kq, pt, ln, 16, 1)[0][0][:, 0].astype(np.int64)
    assert [codes[10], codes[40], codes[46]] == [16, 8, 4]
    bm = sel["block_max"][0, 0]
    assert bm[0] == 127 * max(codes[8:16])          # tokens 8..15 only
    assert bm[1] == 127 * max(codes[16:32])
    assert bm[2] == 127 * max(codes[32:44])         # tokens 44..47 are in the window
    assert bm[3] == INT32_MIN                       # block 3 lies in the window
    assert codes[3] == 127 and codes[50] == 127


def test_no_candidates_when_context_fits_sink_and_window():
    rng = np.random.default_rng(6)
    case = random_case(rng, B=2, hq=4, hkv=1, D=8, lens=(40, 24), page=16)
    d = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=4, k2=4, sink=16, window=24)
    kq, sc, sel, out, lse = run_all(d, case)
    assert sel["n_blocks"].tolist() == [[0], [0]] and sel["n_chunks"].tolist() == [[0], [0]]
    assert (sel["block_idx"] == -1).all()
    od, ld = oracle.dense(d, bf16_bits(case["q"]), bf16_bits(case["k"]), bf16_bits(case["v"]),
                          case["pt"], case["lens"])
    np.testing.assert_allclose(out, od, atol=1e-13)
    np.testing.assert_allclose(lse, ld, atol=1e-13)


# ---------------------------------------------------------------- attention

def _softmax_attention(q, K, V, scale):
    logits = (K.astype(np.float64) @ q.astype(np.float64)) * scale
    return softmax(logits) @ V.astype(np.float64), logsumexp(logits)


@pytest.mark.parametrize("seed", range(3))
def test_dense_matches_library_softmax(seed):
    rng = np.random.default_rng(200 + seed)
    case = random_case(rng, B=2, hq=4, hkv=2, D=8, lens=(37, 70), page=16, perm=True)
    d = dims_for(case, 4, 2, 8)
    out, lse = oracle.dense(d, bf16_bits(case["q"]), bf16_bits(case["k"]), bf16_bits(case["v"]),
                            case["pt"], case["lens"])
    for b in range(2):
        for j in range(4):
            h = j // 2
            o, l = _softmax_attention(case["q"][b, j], case["ks"][b][h], case["vs"][b][h],
                                      1 / math.sqrt(8))
            np.testing.assert_allclose(out[b, j], o, rtol=0, atol=1e-12)
            assert abs(lse[b, j] - l) < 1e-12


def test_sink_and_window_special_case():
    """K1 = K2 = 0 is attention over the sink tokens plus the sliding window."""
    rng = np.random.default_rng(7)
    case = random_case(rng, B=1, hq=4, hkv=1, D=8, lens=(300,), page=16)
    d = dims_for(case, 4, 1, 8, k1=0, k2=0, sink=5, window=23)
    _, _, sel, out, lse = run_all(d, case)
    assert sel["block_idx"].size == 0 and sel["n_blocks"].tolist() == [[0]]
    keep = list(range(5)) + list(range(300 - 23, 300))
    for j in range(4):
        o, l = _softmax_attention(case["q"][0, j], case["ks"][0][0][keep], case["vs"][0][0][keep],
                                  1 / math.sqrt(8))
        np.testing.assert_allclose(out[0, j], o, atol=1e-12)
        assert abs(lse[0, j] - l) < 1e-12


def test_selected_blocks_special_case():
    """The attended set is sink + window + the kept blocks' candidate tokens."""
    rng = np.random.default_rng(8)
    case = random_case(rng, B=1, hq=4, hkv=1, D=8, lens=(333,), page=16)
    d = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=3, k2=4, sink=20, window=30)
    _, _, sel, out, lse = run_all(d, case)
    kept = [k for k in sel["block_idx"][0, 0] if k >= 0]
    assert len(kept) == 4
    toks = set(range(20)) | set(range(303, 333))
    for k in kept:
        toks |= {t for t in range(16 * k, 16 * k + 16) if 20 <= t < 303}
    keep = sorted(toks)
    for j in range(4):
        o, l = _softmax_attention(case["q"][0, j], case["ks"][0][0][keep], case["vs"][0][0][keep],
                                  1 / math.sqrt(8))
        np.testing.assert_allclose(out[0, j], o, atol=1e-12)
        assert abs(lse[0, j] - l) < 1e-12


def test_everything_selected_equals_dense():
    rng = np.random.default_rng(9)
    case = random_case(rng, B=2, hq=8, hkv=2, D=16, lens=(500, 257), page=16, perm=True)
    d = dims_for(case, 8, 2, 16, chunk=64, block=16, k1=100, k2=100, sink=7, window=9)
    _, _, sel, out, lse = run_all(d, case)
    od, ld = oracle.dense(d, bf16_bits(case["q"]), bf16_bits(case["k"]), bf16_bits(case["v"]),
                          case["pt"], case["lens"])
    np.testing.assert_allclose(out, od, atol=1e-12)
    np.testing.assert_allclose(lse, ld, atol=1e-12)
    r = oracle.recall(d, bf16_bits(case["q"]), bf16_bits(case["k"]), case["pt"], case["lens"],
                      sel["block_idx"], sel["n_blocks"])
    np.testing.assert_allclose(r, 1.0, atol=1e-13)


def test_identical_keys_give_the_mean_of_values():
    """All keys equal: the softmax is uniform over the attended set, out is the mean of
    its values and lse = logit + log |T|."""
    rng = np.random.default_rng(10)
    n, D = 200, 8
    key = to_bf16(rng.standard_normal(D))
    ks = [np.tile(key, (1, n, 1)).astype(np.float32)]
    vs = [to_bf16(rng.standard_normal((1, n, D)))]
    kc, pt, ln = paged(ks, 16, 1)
    vc, _, _ = paged(vs, 16, 1)
    q = to_bf16(rng.standard_normal((1, 2, D)))
    d = Dims(1, 2, 1, D, 16, pt.shape[1], kc.shape[0], 32, 16, 0, 0, 10, 15)
    out, lse = oracle.attend(d, bf16_bits(q), bf16_bits(kc), bf16_bits(vc), pt, ln,
                             np.zeros((1, 1, 0), np.int32), np.zeros((1, 1), np.int32))
    keep = list(range(10)) + list(range(185, 200))
    for j in range(2):
        np.testing.assert_allclose(out[0, j], vs[0][0][keep].astype(np.float64).mean(0), atol=1e-13)
        logit = float(np.dot(q[0, j].astype(np.float64), key.astype(np.float64))) / math.sqrt(D)
        assert abs(lse[0, j] - (logit + math.log(len(keep)))) < 1e-12


def test_recall_restriction_identity():
    """R = sum over T of the dense probabilities = exp(lse_T - lse_all), and the sparse
    output is the dense probabilities over T renormalised by R."""
    rng = np.random.default_rng(11)
    case = random_case(rng, B=1, hq=4, hkv=1, D=8, lens=(410,), page=16)
    d = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=4, k2=5, sink=16, window=32)
    _, _, sel, out, lse = run_all(d, case)
    qb, kb = bf16_bits(case["q"]), bf16_bits(case["k"])
    _, ld = oracle.dense(d, qb, kb, bf16_bits(case["v"]), case["pt"], case["lens"])
    r = oracle.recall(d, qb, kb, case["pt"], case["lens"], sel["block_idx"], sel["n_blocks"])
    np.testing.assert_allclose(r, np.exp(lse - ld), rtol=1e-12)
    assert np.all(r > 0) and np.all(r < 1)


def test_tokens_past_the_end_are_ignored():
    """Junk in the slots of a last page past N changes nothing."""
    rng = np.random.default_rng(12)
    case = random_case(rng, B=2, hq=4, hkv=1, D=8, lens=(101, 77), page=16)
    d = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=2, k2=3, sink=4, window=9)
    res1 = run_all(d, case)
    junk = dict(case, k=case["k"].copy(), v=case["v"].copy())
    for b, n in enumerate(case["lens"]):
        pg = case["pt"][b, (n - 1) // 16]
        junk["k"][pg, :, (n % 16):, :] = 96.0
        junk["v"][pg, :, (n % 16):, :] = -96.0
    res2 = run_all(d, junk)
    np.testing.assert_array_equal(res1[1], res2[1])
    for key in ("block_idx", "chunk_idx", "block_max"):
        np.testing.assert_array_equal(res1[2][key], res2[2][key])
    np.testing.assert_array_equal(res1[3], res2[3])


# ------------------------------------------------- block attention mass (cache eviction)

def test_block_mass_is_the_dense_softmax_when_everything_is_kept():
    """Every block kept, no sink or window: the mass of block k for head j is the sum over
    its tokens of scipy's softmax of the dense logits, and each head's masses sum to 1."""
    rng = np.random.default_rng(41)
    case = random_case(rng, B=2, hq=4, hkv=2, D=16, lens=(150, 97), page=16, perm=True)
    d = dims_for(case, 4, 2, 16, chunk=32, block=16, k1=100, k2=100, sink=0, window=0)
    _, _, sel, _, _ = run_all(d, case)
    m = oracle.block_mass(d, bf16_bits(case["q"]), bf16_bits(case["k"]), case["pt"], case["lens"],
                          sel["block_idx"], sel["n_blocks"])
    for b, n in enumerate(case["lens"]):
        for j in range(4):
            keys = case["ks"][b][j // 2].astype(np.float64)              # [n][D]
            p = softmax(keys @ case["q"][b, j].astype(np.float64) / 4.0)
            want = np.zeros(d.max_blocks)
            np.add.at(want, np.arange(n) // 16, p)
            np.testing.assert_allclose(m[b, j], want, atol=1e-13)
            assert abs(m[b, j].sum() - 1.0) < 1e-12


def test_block_mass_identical_keys_is_token_count_over_t():
    """All keys equal: the softmax is uniform over T, so block k receives |T n k| / |T|
    (sink 10 and window 15 cut blocks 0 and 11 short)."""
    rng = np.random.default_rng(42)
    n, D = 200, 8
    key = to_bf16(rng.standard_normal(D))
    kc, pt, ln = paged([np.tile(key, (1, n, 1)).astype(np.float32)], 16, 1)
    q = to_bf16(rng.standard_normal((1, 2, D)))
    d = Dims(1, 2, 1, D, 16, pt.shape[1], kc.shape[0], 32, 16, 0, 2, 10, 15)
    bidx = np.array([[[3, 7]]], np.int32)
    m = oracle.block_mass(d, bf16_bits(q), bf16_bits(kc), pt, ln, bidx, np.array([[2]], np.int32))
    want = np.zeros(d.max_blocks)
    want[0] = 10            # sink: tokens 0..9
    want[3] = want[7] = 16  # kept blocks, inside the candidate region [10, 185)
    want[11] = 7            # window: tokens 185..199 -> block 11 holds 185..191
    want[12] = 8            # and block 12 holds 192..199
    want /= want.sum()      # |T| = 10 + 32 + 15 = 57
    for j in range(2):
        np.testing.assert_allclose(m[0, j], want, atol=1e-14)


def test_block_mass_restriction_identity():
    """Mass over the sparse set T = dense mass / recall on T's blocks, zero elsewhere (sink
    and window are whole blocks here, so every block is in T entirely or not at all)."""
    rng = np.random.default_rng(43)
    case = random_case(rng, B=1, hq=4, hkv=1, D=8, lens=(410,), page=16)
    d = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=4, k2=5, sink=16, window=26)
    _, _, sel, _, _ = run_all(d, case)
    qb, kb = bf16_bits(case["q"]), bf16_bits(case["k"])
    ms = oracle.block_mass(d, qb, kb, case["pt"], case["lens"], sel["block_idx"], sel["n_blocks"])
    every = np.arange(d.max_blocks, dtype=np.int32)[None, None, :]
    dd = dims_for(case, 4, 1, 8, chunk=32, block=16, k1=d.max_blocks, k2=d.max_blocks, sink=0,
                  window=0)
    md = oracle.block_mass(dd, qb, kb, case["pt"], case["lens"], every,
                           np.array([[d.max_blocks]], np.int32))
    r = oracle.recall(d, qb, kb, case["pt"], case["lens"], sel["block_idx"], sel["n_blocks"])
    in_t = {0, 24, 25}   # sink: block 0; window: tokens 384..409
    in_t |= {int(k) for k in sel["block_idx"][0, 0, : sel["n_blocks"][0, 0]]}
    for j in range(4):
        for k in range(d.max_blocks):
            if k in in_t:
                assert abs(ms[0, j, k] * r[0, j] - md[0, j, k]) < 1e-13
            else:
                assert ms[0, j, k] == 0.0
