"""Pins of the float64 oracle to facts outside itself (CPU only).

Each check is chosen so that a plausible slip in the oracle -- a dropped
term, a wrong sign or index, a transposed operand, a wrong rounding rule --
fails at least one of them:

  * element formats against independent library decoders (numpy float16,
    torch bfloat16 / float8_e4m3fn) over every code;
  * E4M3 encoding: round trip, ties to even at every midpoint, saturation,
    and agreement with torch's cast inside the finite range;
  * decode attention against numpy softmax(q K^T * scale) V on the gathered
    contiguous K/V (library matmul), against 50-digit ``decimal`` brute force
    on tiny inputs, invariance under relabelling physical blocks, and the
    closed forms (one token returns its value row; identical keys return the
    mean of V; a dominant key returns its value; equal queries in a GQA group
    give equal rows; length 0 gives zeros);
  * split-K partials + log-sum-exp merge equal the unsplit result;
  * causal paged prefill against torch softmax(Q K^T * scale + causal mask) V
    on the gathered keys, 50-digit brute force, decode for one-token chunks,
    one pass against two chunks, block relabelling, and the first prompt
    token returning its own value;
  * append / copy_blocks checked by reading back through the block table.
"""
import decimal
import math

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(12345)


def bits16(x, dtype):
    t = torch.from_numpy(np.asarray(x, np.float32)).to({"f16": torch.float16, "bf16": torch.bfloat16}[dtype])
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_e4m3(x):
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


# ------------------------------------------------------------------ formats
def test_f16_decode_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = oracle.dequantize(codes, "f16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decode_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.dequantize(codes, "bf16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.dequantize(codes, "e4m3")
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7f and 0xff only
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_round_trip_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_to_double(c)) == c


def test_e4m3_encode_ties_to_even_at_every_midpoint():
    vals = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    for c in range(0x7E):
        mid = (vals[c] + vals[c + 1]) / 2  # exact in float32 (few significant bits)
        assert np.float32(mid) == mid
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == want
        assert oracle.e4m3_encode(-mid) == want | 0x80
        # just off the midpoint goes to the nearer code
        lo = np.nextafter(np.float32(mid), np.float32(0))
        hi = np.nextafter(np.float32(mid), np.float32(1e9))
        assert oracle.e4m3_encode(lo) == c
        assert oracle.e4m3_encode(hi) == c + 1


def test_e4m3_encode_saturates():
    for x in (448.0, 449.0, 464.0, 465.0, 1e6, 3.0e38):
        assert oracle.e4m3_encode(x) == 0x7E
        assert oracle.e4m3_encode(-x) == 0xFE


def test_e4m3_encode_matches_torch_inside_the_range():
    x = np.concatenate([RNG.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 0.05, 1.0, 30.0, 120.0)])
    x = x[np.abs(x) < 448.0]
    ref = bits_e4m3(x)
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], np.uint8)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- attention
def make_case(S, Hq, Hkv, D, lens, NB=None, dtype="f16", seed=0, identity=False):
    rng = np.random.default_rng(seed)
    b = 16
    need = sum(-(-L // b) for L in lens)
    NB = NB or need + 3
    k = rng.standard_normal((NB, Hkv, b, D)).astype(np.float32)
    v = rng.standard_normal((NB, Hkv, b, D)).astype(np.float32)
    q = rng.standard_normal((S, Hq, D)).astype(np.float32)
    MB = max(1, max(-(-L // b) for L in lens))
    bt = np.full((S, MB), -1, np.int32)
    ids = np.arange(NB) if identity else rng.permutation(NB)
    pos = 0
    for s, L in enumerate(lens):
        n = -(-L // b)
        bt[s, :n] = ids[pos:pos + n]
        pos += n
    conv = (lambda a: bits16(a, dtype)) if dtype != "e4m3" else bits_e4m3
    qd = "f16" if dtype == "f16" else "bf16"
    return dict(q=bits16(q, qd), q_dtype=qd, k_pool=conv(k), v_pool=conv(v), kv_dtype=dtype,
                block_tables=bt, seq_lens=np.array(lens, np.int32), scale=1 / math.sqrt(D))


def gathered(case, s, h):
    b = 16
    L = int(case["seq_lens"][s])
    K = np.stack([case["k_pool"][case["block_tables"][s, t // b], h, t % b] for t in range(L)]) if L else None
    V = np.stack([case["v_pool"][case["block_tables"][s, t // b], h, t % b] for t in range(L)]) if L else None
    return K, V


@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("G", [1, 4])
def test_decode_matches_contiguous_library_attention(dtype, G):
    Hkv = 2
    case = make_case(3, Hkv * G, Hkv, 32, [5, 40, 33], dtype=dtype, seed=1)
    ks, vs = (0.05, 0.07) if dtype == "e4m3" else (1.0, 1.0)
    out = oracle.paged_decode(**case, k_scale=ks, v_scale=vs)
    qf = oracle.dequantize(case["q"], case["q_dtype"])
    for s in range(3):
        for i in range(Hkv * G):
            K, V = gathered(case, s, i // G)
            Kf = torch.from_numpy(oracle.dequantize(K, dtype) * ks)
            Vf = torch.from_numpy(oracle.dequantize(V, dtype) * vs)
            qi = torch.from_numpy(qf[s, i])
            ref = torch.softmax((Kf @ qi) * case["scale"], dim=0) @ Vf
            assert np.max(np.abs(out[s, i] - ref.numpy())) <= 1e-12


def test_decode_matches_50_digit_brute_force():
    case = make_case(2, 2, 1, 8, [13, 20], dtype="bf16", seed=2)
    out = oracle.paged_decode(**case)
    decimal.getcontext().prec = 50
    D = decimal.Decimal
    qf = oracle.dequantize(case["q"], "bf16")
    for s in range(2):
        K, V = gathered(case, s, 0)
        Kf, Vf = oracle.dequantize(K, "bf16"), oracle.dequantize(V, "bf16")
        for i in range(2):
            sc = [sum(D(float(qf[s, i, d])) * D(float(Kf[t, d])) for d in range(8)) * D(case["scale"])
                  for t in range(len(Kf))]
            m = max(sc)
            w = [(x - m).exp() for x in sc]
            tot = sum(w)
            for d in range(8):
                ref = sum(w[t] * D(float(Vf[t, d])) for t in range(len(w))) / tot
                assert abs(out[s, i, d] - float(ref)) <= 1e-13


def test_decode_invariant_under_block_relabelling():
    case = make_case(4, 8, 2, 64, [1, 17, 50, 64], NB=40, dtype="f16", seed=3)
    out = oracle.paged_decode(**case)
    perm = np.random.default_rng(9).permutation(40)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(40)
    case2 = dict(case)
    case2["k_pool"] = case["k_pool"][inv]
    case2["v_pool"] = case["v_pool"][inv]
    bt = case["block_tables"]
    case2["block_tables"] = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode(**case2)
    assert np.array_equal(out, out2)


def test_closed_form_one_token_returns_its_value():
    case = make_case(2, 4, 2, 16, [1, 1], dtype="bf16", seed=4)
    out = oracle.paged_decode(**case)
    for s in range(2):
        for i in range(4):
            _, V = gathered(case, s, i // 2)
            assert np.array_equal(out[s, i], oracle.dequantize(V[0], "bf16"))


def test_closed_form_identical_keys_give_mean_value():
    case = make_case(1, 2, 1, 16, [37], dtype="bf16", seed=5)
    kp = case["k_pool"].copy()
    kp[:] = kp[0, 0, 0]
    case["k_pool"] = kp
    out = oracle.paged_decode(**case)
    _, V = gathered(case, 0, 0)
    ref = oracle.dequantize(V, "bf16").mean(axis=0)
    assert np.max(np.abs(out[0] - ref)) <= 1e-12


def test_closed_form_dominant_key_selects_its_value():
    case = make_case(1, 1, 1, 16, [29], dtype="bf16", seed=6)
    qf = oracle.dequantize(case["q"], "bf16")[0, 0]
    kp = case["k_pool"].copy()
    bt = case["block_tables"]
    t = 21
    kp[bt[0, t // 16], 0, t % 16] = bits16((qf * 50).astype(np.float32), "bf16")
    case["k_pool"] = kp
    out = oracle.paged_decode(**case)
    _, V = gathered(case, 0, 0)
    assert np.max(np.abs(out[0, 0] - oracle.dequantize(V[t], "bf16"))) < 1e-6


def test_gqa_equal_queries_give_equal_rows_and_zero_length_gives_zeros():
    case = make_case(2, 8, 2, 32, [45, 0], dtype="f16", seed=7)
    q = case["q"].copy()
    q[0, 4:8] = q[0, 4]
    case["q"] = q
    out = oracle.paged_decode(**case)
    for i in range(5, 8):
        assert np.array_equal(out[0, i], out[0, 4])
    assert not np.array_equal(out[0, 3], out[0, 4])
    assert np.all(out[1] == 0.0)


@pytest.mark.parametrize("P", [16, 32, 48, 512])
def test_partitioned_merge_equals_unsplit(P):
    case = make_case(3, 4, 2, 32, [1, 70, 130], dtype="bf16", seed=8)
    out = oracle.paged_decode(**case)
    m, l, o = oracle.paged_decode_partials(**case, partition_tokens=P)
    merged = oracle.lse_merge(m, l, o)
    assert np.max(np.abs(merged - out)) <= 1e-12


def test_oracle_rejects_out_of_pool_block_ids():
    case = make_case(1, 1, 1, 16, [20], NB=4, dtype="bf16", seed=10)
    case["block_tables"] = case["block_tables"].copy()
    case["block_tables"][0, 1] = 4
    with pytest.raises(ValueError):
        oracle.paged_decode(**case)


# ------------------------------------------------------------------ prefill
def make_prefill_case(Hq, Hkv, D, lens, qlens, dtype="bf16", seed=0, NB=None):
    """A decode-style case plus packed query rows: sequence s owns the last
    qlens[s] of its lens[s] positions, rows query_start[s]..query_start[s+1]."""
    case = make_case(len(lens), Hq, Hkv, D, lens, dtype=dtype, seed=seed, NB=NB)
    rng = np.random.default_rng(seed + 100)
    T = int(sum(qlens))
    qd = case["q_dtype"]
    case["q"] = bits16(rng.standard_normal((T, Hq, D)).astype(np.float32), qd)
    case["query_start"] = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    return case


def causal_reference(case, G, ks=1.0, vs=1.0):
    """torch float64 softmax(Q K^T * scale + causal mask) V per sequence, on the
    gathered contiguous keys and values."""
    qf = oracle.dequantize(case["q"], case["q_dtype"])
    T, Hq, D = qf.shape
    out = np.zeros((T, Hq, D))
    qs = case["query_start"]
    for s in range(len(case["seq_lens"])):
        L = int(case["seq_lens"][s])
        n = int(qs[s + 1] - qs[s])
        if n == 0:
            continue
        ctx = L - n
        pos = torch.arange(ctx, L, dtype=torch.int64)[:, None]
        key = torch.arange(L, dtype=torch.int64)[None, :]
        mask = key > pos
        for h in range(Hq // G):
            K, V = gathered(case, s, h)
            Kf = torch.from_numpy(oracle.dequantize(K, case["kv_dtype"]) * ks)
            Vf = torch.from_numpy(oracle.dequantize(V, case["kv_dtype"]) * vs)
            for g in range(G):
                i = h * G + g
                Q = torch.from_numpy(qf[qs[s]:qs[s + 1], i])
                sc = (Q @ Kf.T) * case["scale"]
                sc = sc.masked_fill(mask, float("-inf"))
                out[qs[s]:qs[s + 1], i] = (torch.softmax(sc, dim=1) @ Vf).numpy()
    return out


@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("G", [1, 4])
def test_prefill_matches_contiguous_causal_library_attention(dtype, G):
    Hkv = 2
    case = make_prefill_case(Hkv * G, Hkv, 32, [5, 40, 33, 70], [5, 17, 1, 33], dtype=dtype, seed=11)
    ks, vs = (0.05, 0.07) if dtype == "e4m3" else (1.0, 1.0)
    out = oracle.paged_prefill(**case, k_scale=ks, v_scale=vs)
    ref = causal_reference(case, G, ks, vs)
    assert np.max(np.abs(out - ref)) <= 1e-12


def test_prefill_of_single_tokens_equals_decode():
    case = make_prefill_case(8, 2, 32, [1, 17, 50, 64], [1, 1, 1, 1], dtype="bf16", seed=12)
    pre = oracle.paged_prefill(**case)
    dec_case = {k: v for k, v in case.items() if k != "query_start"}
    dec = oracle.paged_decode(**dec_case)
    assert np.max(np.abs(pre - dec)) <= 1e-14


def test_prefill_first_prompt_token_returns_its_value():
    case = make_prefill_case(4, 2, 16, [9, 30], [9, 30], dtype="bf16", seed=13)
    out = oracle.paged_prefill(**case)
    for s in range(2):
        row = case["query_start"][s]
        for i in range(4):
            _, V = gathered(case, s, i // 2)
            assert np.array_equal(out[row, i], oracle.dequantize(V[0], "bf16"))


def test_prefill_in_two_chunks_equals_one_pass():
    whole = make_prefill_case(4, 1, 16, [50], [50], dtype="bf16", seed=14)
    out = oracle.paged_prefill(**whole)
    first = dict(whole, q=whole["q"][:20], query_start=np.array([0, 20], np.int32),
                 seq_lens=np.array([20], np.int32))
    second = dict(whole, q=whole["q"][20:], query_start=np.array([0, 30], np.int32))
    a = oracle.paged_prefill(**first)
    b = oracle.paged_prefill(**second)
    assert np.max(np.abs(np.concatenate([a, b]) - out)) <= 1e-15


def test_prefill_matches_50_digit_brute_force():
    case = make_prefill_case(2, 1, 8, [13, 20], [4, 6], dtype="bf16", seed=15)
    out = oracle.paged_prefill(**case)
    decimal.getcontext().prec = 50
    D = decimal.Decimal
    qf = oracle.dequantize(case["q"], "bf16")
    qs = case["query_start"]
    for s in range(2):
        K, V = gathered(case, s, 0)
        Kf, Vf = oracle.dequantize(K, "bf16"), oracle.dequantize(V, "bf16")
        L = len(Kf)
        n = qs[s + 1] - qs[s]
        for j in range(n):
            p = L - n + j
            for i in range(2):
                row = qf[qs[s] + j, i]
                sc = [sum(D(float(row[d])) * D(float(Kf[t, d])) for d in range(8)) * D(case["scale"])
                      for t in range(p + 1)]
                m = max(sc)
                w = [(x - m).exp() for x in sc]
                tot = sum(w)
                for d in range(8):
                    ref = sum(w[t] * D(float(Vf[t, d])) for t in range(len(w))) / tot
                    assert abs(out[qs[s] + j, i, d] - float(ref)) <= 1e-13


def test_prefill_invariant_under_block_relabelling():
    case = make_prefill_case(8, 2, 64, [1, 17, 50, 64], [1, 10, 50, 3], NB=40, dtype="f16", seed=16)
    out = oracle.paged_prefill(**case)
    perm = np.random.default_rng(19).permutation(40)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(40)
    bt = case["block_tables"]
    case2 = dict(case, k_pool=case["k_pool"][inv], v_pool=case["v_pool"][inv],
                 block_tables=np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32))
    assert np.array_equal(out, oracle.paged_prefill(**case2))


def test_prefill_rejects_more_new_tokens_than_the_sequence_holds():
    case = make_prefill_case(2, 1, 16, [10], [10], dtype="bf16", seed=17)
    case["seq_lens"] = np.array([9], np.int32)
    with pytest.raises(ValueError):
        oracle.paged_prefill(**case)


# ------------------------------------------------------------ append / copy
@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
def test_append_lands_at_the_mapped_slot_only(dtype):
    NB, Hkv, D = 6, 2, 32
    rng = np.random.default_rng(11)
    conv = (lambda a: bits16(a, dtype)) if dtype != "e4m3" else bits_e4m3
    kp = conv(rng.standard_normal((NB, Hkv, 16, D)).astype(np.float32))
    vp = conv(rng.standard_normal((NB, Hkv, 16, D)).astype(np.float32))
    in_dt = dtype if dtype != "e4m3" else "bf16"
    kn = bits16(rng.standard_normal((4, Hkv, D)).astype(np.float32) * 3, in_dt)
    vn = bits16(rng.standard_normal((4, Hkv, D)).astype(np.float32) * 3, in_dt)
    slots = np.array([5 * 16 + 3, -1, 0, 2 * 16 + 15], np.int64)
    k2, v2 = kp.copy(), vp.copy()
    ks, vs = (0.02, 0.03) if dtype == "e4m3" else (1.0, 1.0)
    oracle.append(kn, vn, in_dt, slots, k2, v2, dtype, ks, vs)
    touched = np.zeros((NB, 16), bool)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        blk, off = sl // 16, sl % 16
        touched[blk, off] = True
        if dtype == "e4m3":
            xk = oracle.dequantize(kn[t], "bf16").astype(np.float32) / np.float32(ks)
            assert np.array_equal(k2[blk, :, off], bits_e4m3(xk))
            xv = oracle.dequantize(vn[t], "bf16").astype(np.float32) / np.float32(vs)
            assert np.array_equal(v2[blk, :, off], bits_e4m3(xv))
        else:
            assert np.array_equal(k2[blk, :, off], kn[t]) and np.array_equal(v2[blk, :, off], vn[t])
    for blk in range(NB):
        for off in range(16):
            if not touched[blk, off]:
                assert np.array_equal(k2[blk, :, off], kp[blk, :, off])
                assert np.array_equal(v2[blk, :, off], vp[blk, :, off])


def test_copy_blocks_copies_pairs_and_nothing_else():
    rng = np.random.default_rng(12)
    kp = rng.integers(0, 65535, size=(8, 2, 16, 16), dtype=np.uint16)
    vp = rng.integers(0, 65535, size=(8, 2, 16, 16), dtype=np.uint16)
    k2, v2 = kp.copy(), vp.copy()
    oracle.copy_blocks(k2, v2, "bf16", [[1, 6], [3, 0]])
    assert np.array_equal(k2[6], kp[1]) and np.array_equal(v2[6], vp[1])
    assert np.array_equal(k2[0], kp[3]) and np.array_equal(v2[0], vp[3])
    for blk in (1, 2, 3, 4, 5, 7):
        assert np.array_equal(k2[blk], kp[blk]) and np.array_equal(v2[blk], vp[blk])
