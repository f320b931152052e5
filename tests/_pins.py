"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.  Each pin takes ``mutant`` (0 = the real
oracle; >0 = a planted-mistake build used by the mutation test) and raises
AssertionError when the oracle violates it.

Citations name the page and section of the exact_attention_online pages:
  [blog]  FlashAttention (NeurIPS 2022) summary blog
  [fa2]   FlashAttention-2 review thread
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_qkv(B, H, Hkv, N, d, seed, dout=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, Hkv, N, d))
    v = rng.standard_normal((B, Hkv, N, d))
    if dout:
        return q, k, v, rng.standard_normal((B, H, N, d))
    return q, k, v


def torch_attention(q, k, v, causal, scale):
    """Library special case: torch fp64 CPU matmul + softmax (+ logsumexp)."""
    q, k, v = (torch.as_tensor(x, dtype=torch.float64) for x in (q, k, v))
    G = q.shape[1] // k.shape[1]
    k = k.repeat_interleave(G, dim=1)
    v = v.repeat_interleave(G, dim=1)
    s = (q @ k.transpose(-1, -2)) * scale
    if causal:
        N = q.shape[2]
        mask = torch.ones(N, N, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, float("-inf"))
    return torch.softmax(s, dim=-1) @ v, torch.logsumexp(s, dim=-1)


# ---------------------------------------------------------------- forward pins

def pin_rows_sum_to_one(mutant=0):
    """[blog] "(Safe) Softmax": every row of P is a probability vector; with
    the causal mask, P_ij = 0 for j > i."""
    for causal in (False, True):
        q, k, v = rand_qkv(1, 2, 1, 37, 8, seed=11)
        _, _, p = oracle.attn_fwd(q, k, v, causal, 0.35, return_p=True, mutant=mutant)
        assert np.all(p >= 0)
        assert np.max(np.abs(p.sum(-1) - 1.0)) <= 1e-12, "rows of P must sum to 1"
        if causal:
            assert np.all(np.triu(p[0, 0], 1) == 0) and np.all(np.triu(p[0, 1], 1) == 0)


def pin_torch_library(mutant=0):
    """[blog] "From Online Softmax to FlashAttention": standard attention
    S = QK^T*scale, P = softmax(S), O = PV equals torch's fp64 matmul/softmax
    and its scaled_dot_product_attention (math kernel, GQA by
    repeat_interleave); LSE equals torch.logsumexp of the scaled scores."""
    for (B, H, Hkv, N, d, causal) in [(2, 4, 2, 33, 16, True), (1, 3, 3, 20, 8, False),
                                      (1, 4, 1, 65, 32, True)]:
        q, k, v = rand_qkv(B, H, Hkv, N, d, seed=N)
        scale = 1 / math.sqrt(d)
        o, lse = oracle.attn_fwd(q, k, v, causal, scale, mutant=mutant)
        to, tl = torch_attention(q, k, v, causal, scale)
        assert np.max(np.abs(o - to.numpy())) <= 1e-12
        assert np.max(np.abs(lse - tl.numpy())) <= 1e-12
        tq, tk, tv = (torch.as_tensor(x) for x in (q, k, v))
        sd = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=causal, scale=scale, enable_gqa=(H != Hkv))
        assert np.max(np.abs(o - sd.numpy())) <= 1e-12


def pin_online_matches_three_pass(mutant=0):
    """[blog] "Online Softmax" (d_N = d'_N) and "FlashAttention" (o_N = o'_N,
    tiles of b keys); [fa2] deferred division by l.  Both one-pass forms agree
    with the three-loop safe softmax to 1e-12 relative."""
    q, k, v = rand_qkv(2, 2, 1, 70, 16, seed=5)
    q *= 3.0  # wide score range, so rescaling really happens
    for causal in (False, True):
        o3, l3 = oracle.attn_fwd(q, k, v, causal, 0.5, mutant=mutant)
        for block in (1, 7, 64, 128):
            for deferred in (False, True):
                o1, l1 = oracle.attn_fwd_online(q, k, v, causal, 0.5, block, deferred,
                                                mutant=mutant)
                rel = np.max(np.abs(o1 - o3)) / np.max(np.abs(o3))
                assert rel <= 1e-12, (block, deferred, rel)
                assert np.max(np.abs(l1 - l3)) <= 1e-12 * np.max(np.abs(l3))


def pin_identical_keys(mutant=0):
    """Closed form: if every key is the same vector k, all visible scores of a
    row are equal, so O_i is the plain mean of the visible V rows and
    LSE_i = scale*<q_i,k> + ln(#visible)."""
    rng = np.random.default_rng(3)
    N, d, scale = 29, 8, 0.7
    kk = rng.standard_normal(d)
    q = rng.standard_normal((1, 1, N, d))
    k = np.broadcast_to(kk, (1, 1, N, d)).copy()
    v = rng.standard_normal((1, 1, N, d))
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, scale, mutant=mutant)
        for i in range(N):
            cnt = i + 1 if causal else N
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, :cnt].mean(0))) <= 1e-13
            want = scale * float(q[0, 0, i] @ kk) + math.log(cnt)
            assert abs(lse[0, 0, i] - want) <= 1e-13


def pin_one_hot(mutant=0):
    """Closed form: Q_i = e_i and K_j = a*e_pi(j) give s_ij = a*scale when
    pi(j) = i and 0 otherwise, so O_i = (E v_{pi^-1(i)} + sum_{j != pi^-1(i)} v_j)
    / (E + N - 1) with E = exp(a*scale); for large a this selects one V row."""
    N = d = 12
    rng = np.random.default_rng(4)
    perm = rng.permutation(N)
    inv = np.argsort(perm)
    q = np.eye(N)[None, None]
    v = rng.standard_normal((1, 1, N, d))
    for a, tol in ((2.0, 1e-13), (400.0, 1e-13)):
        k = (a * np.eye(N)[perm])[None, None]
        o, lse = oracle.attn_fwd(q, k, v, False, 0.25, mutant=mutant)
        E = math.exp(a * 0.25)
        for i in range(N):
            sel = inv[i]
            want = (E * v[0, 0, sel] + v[0, 0].sum(0) - v[0, 0, sel]) / (E + N - 1)
            assert np.max(np.abs(o[0, 0, i] - want)) <= tol * max(1.0, np.abs(want).max())
            assert abs(lse[0, 0, i] - math.log(E + N - 1)) <= 1e-12
        if a > 100:
            assert np.max(np.abs(o[0, 0] - v[0, 0, inv])) <= 1e-12


def pin_causal_row0_and_single_key(mutant=0):
    """Special cases: with the causal mask, query 0 sees only key 0, so O_0 = V_0
    and LSE_0 = scale*<q_0,k_0>; with N = 1 the same holds without a mask."""
    q, k, v = rand_qkv(1, 2, 2, 19, 8, seed=8)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.4, mutant=mutant)
    for h in range(2):
        assert np.array_equal(o[0, h, 0], v[0, h, 0])
        assert abs(lse[0, h, 0] - 0.4 * float(q[0, h, 0] @ k[0, h, 0])) <= 1e-14
    q1, k1, v1 = q[:, :, :1], k[:, :, :1], v[:, :, :1]
    o, lse = oracle.attn_fwd(q1, k1, v1, False, 0.4, mutant=mutant)
    assert np.array_equal(o[0, :, 0], v1[0, :, 0])


def pin_shift_invariance(mutant=0):
    """Invariance: adding one vector u to every key adds scale*<q_i,u> to every
    score of row i, which softmax ignores: O, dQ and dV are unchanged and LSE_i
    moves by scale*<q_i,u>."""
    q, k, v, do = rand_qkv(1, 2, 1, 24, 8, seed=9, dout=True)
    u = np.random.default_rng(10).standard_normal(8)
    for causal in (False, True):
        o0, l0 = oracle.attn_fwd(q, k, v, causal, 0.3, mutant=mutant)
        o1, l1 = oracle.attn_fwd(q, k + u, v, causal, 0.3, mutant=mutant)
        assert np.max(np.abs(o1 - o0)) <= 1e-12
        assert np.max(np.abs(l1 - l0 - 0.3 * (q @ u))) <= 1e-12
        g0 = oracle.attn_bwd(q, k, v, do, causal, 0.3, mutant=mutant)
        g1 = oracle.attn_bwd(q, k + u, v, do, causal, 0.3, mutant=mutant)
        assert np.max(np.abs(g1[0] - g0[0])) <= 1e-11
        assert np.max(np.abs(g1[2] - g0[2])) <= 1e-12


def pin_golden_closed_form(mutant=0):
    """tests/golden/closed_form.json: integer score exponentials, exact
    rational O and exp(LSE) (see make_closed_form.py)."""
    with open(os.path.join(GOLDEN, "closed_form.json")) as f:
        data = json.load(f)
    for c in data["cases"]:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        o, lse = oracle.attn_fwd(q, k, v, c["causal"], c["scale"], mutant=mutant)
        want_o = np.vectorize(lambda s: float(Fraction(s)))(np.array(c["o_exact"]))
        want_l = np.vectorize(lambda s: math.log(Fraction(s)))(np.array(c["lse_exp_exact"]))
        assert np.max(np.abs(o - want_o)) <= 1e-13, c["name"]
        assert np.max(np.abs(lse - want_l)) <= 1e-13, c["name"]


# --------------------------------------------------------------- backward pins

def _loss_and_grads(q, k, v, w, causal, scale, mutant):
    o, _ = oracle.attn_fwd(q, k, v, causal, scale, mutant=mutant)
    return float((o * w).sum())


def pin_finite_differences(mutant=0):
    """Central finite differences (h = 1e-6, fp64) of L = sum(O * W) equal the
    analytic dQ, dK, dV with dO = W (relative error <= 1e-6), on tiny MHA and
    GQA cases with and without the causal mask."""
    for (H, Hkv, N, d, causal) in [(2, 1, 9, 4, True), (1, 1, 16, 8, False), (2, 2, 7, 3, True)]:
        q, k, v, w = rand_qkv(1, H, Hkv, N, d, seed=100 + N, dout=True)
        scale = 1 / math.sqrt(d)
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, w, causal, scale, mutant=mutant)
        h = 1e-6
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            it = np.nditer(x, flags=["multi_index"])
            for _ in it:
                idx = it.multi_index
                old = x[idx]
                x[idx] = old + h
                lp = _loss_and_grads(q, k, v, w, causal, scale, mutant)
                x[idx] = old - h
                lm = _loss_and_grads(q, k, v, w, causal, scale, mutant)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            rel = np.linalg.norm(num - g) / max(np.linalg.norm(num), 1e-300)
            assert rel <= 1e-6, (name, H, Hkv, N, d, causal, rel)


def pin_torch_autograd(mutant=0):
    """Library special case: torch fp64 autograd through matmul/softmax gives the
    same dQ, dK, dV (GQA through repeat_interleave, whose backward sums the
    group)."""
    for (B, H, Hkv, N, d, causal) in [(1, 4, 2, 40, 16, True), (2, 2, 2, 33, 8, False)]:
        q, k, v, do = rand_qkv(B, H, Hkv, N, d, seed=200 + N, dout=True)
        scale = 1 / math.sqrt(d)
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, scale, mutant=mutant)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        o, _ = torch_attention(tq, tk, tv, causal, scale)
        o.backward(torch.as_tensor(do))
        for mine, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.max(np.abs(mine - ref.numpy())) <= 1e-11


def pin_backward_invariants(mutant=0):
    """Invariants of the gradients: rows of P sum to 1, so sum_j dV_j equals the
    sum of dO over the group's query rows; sum_j dS_ij = 0, so sum_j dK_j = 0;
    and D_i = <dO_i, O_i> equals rowsum(P o dP) with dP = dO V^T."""
    for causal in (False, True):
        B, H, Hkv, N, d = 1, 4, 2, 31, 8
        q, k, v, do = rand_qkv(B, H, Hkv, N, d, seed=300, dout=True)
        dq, dk, dv, D = oracle.attn_bwd(q, k, v, do, causal, 0.4, mutant=mutant)
        G = H // Hkv
        for g in range(Hkv):
            want = do[0, g * G:(g + 1) * G].sum(axis=(0, 1))
            assert np.max(np.abs(dv[0, g].sum(0) - want)) <= 1e-12
            assert np.max(np.abs(dk[0, g].sum(0))) <= 1e-12
        _, _, p = oracle.attn_fwd(q, k, v, causal, 0.4, return_p=True, mutant=mutant)
        vr = np.repeat(v, G, axis=1)
        dp = do @ vr.transpose(0, 1, 3, 2)
        assert np.max(np.abs((p * dp).sum(-1) - D)) <= 1e-12


def pin_gqa_equals_repeated_mha(mutant=0):
    """GQA/MQA: query head h uses key/value head h / (H/Hkv); the result equals
    MHA on K, V repeated per group, and dK, dV equal the group sums of the MHA
    gradients."""
    B, H, Hkv, N, d = 1, 6, 2, 18, 8
    q, k, v, do = rand_qkv(B, H, Hkv, N, d, seed=400, dout=True)
    G = H // Hkv
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.3, mutant=mutant)
        om, lm = oracle.attn_fwd(q, kr, vr, causal, 0.3, mutant=mutant)
        assert np.max(np.abs(o - om)) <= 1e-14 and np.max(np.abs(lse - lm)) <= 1e-14
        dq, dk, dv, _ = oracle.attn_bwd(q, k, v, do, causal, 0.3, mutant=mutant)
        dqm, dkm, dvm, _ = oracle.attn_bwd(q, kr, vr, do, causal, 0.3, mutant=mutant)
        assert np.max(np.abs(dq - dqm)) <= 1e-13
        assert np.max(np.abs(dk - dkm.reshape(B, Hkv, G, N, d).sum(2))) <= 1e-12
        assert np.max(np.abs(dv - dvm.reshape(B, Hkv, G, N, d).sum(2))) <= 1e-12


def pin_row_subset(mutant=0):
    """The row-subset entry point returns exactly the rows of the full result."""
    q, k, v = rand_qkv(2, 2, 1, 21, 8, seed=500)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.3, mutant=mutant)
    rows = np.array([0, 5, 20, 21, 42, 83])
    os_, ls = oracle.attn_fwd(q, k, v, True, 0.3, rows=rows, mutant=mutant)
    assert np.array_equal(os_, o.reshape(-1, 8)[rows])
    assert np.array_equal(ls, lse.reshape(-1)[rows])


# ------------------------------------------------------------------- FP8
# The e4m3 format as defined (FlashAttention-3 summary names FP8 and block
# quantization; the format itself is fixed by its definition): sign, 4 exponent
# bits with bias 7, 3 mantissa bits, subnormals m * 2^-9, no infinities,
# S.1111.111 = NaN, largest finite magnitude 448.

def _e4m3_value_by_definition(code):
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return math.nan
    v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -v if s else v


def pin_e4m3_definition(mutant=0):
    """Values fixed by the format: 1.0, the largest finite 448, the smallest
    subnormal 2^-9, the smallest normal 2^-6, zero and negative zero, a
    subnormal, ties to the even mantissa, saturation beyond 448."""
    want = {1.0: 0x38, 448.0: 0x7E, -448.0: 0xFE, 2.0 ** -9: 0x01, 2.0 ** -6: 0x08,
            7 * 2.0 ** -9: 0x07, 0.0: 0x00, -1.5: 0xBC, 240.0: 0x77,
            1.0625: 0x38,           # midway 1 (m=0) / 1.125 (m=1): even m=0
            1.1875: 0x3A,           # midway 1.125 (m=1) / 1.25 (m=2): even m=2
            1.5 * 2.0 ** -9: 0x02,  # midway 1 and 2 subnormal steps: even 2
            460.0: 0x7E, 1000.0: 0x7E, -1e6: 0xFE}
    for x, c in want.items():
        got = oracle.e4m3_encode(x, mutant)
        assert got == c, (x, hex(got), hex(c))
    assert oracle.e4m3_encode(-0.0, mutant) == 0x80


def pin_e4m3_nearest(mutant=0):
    """Brute force: every finite code round-trips, and random values encode
    to the nearest finite value (ties to the even mantissa; beyond 448: 448)."""
    vals = np.array([_e4m3_value_by_definition(c) for c in range(256)])
    finite = [c for c in range(256) if not math.isnan(vals[c])]
    for c in finite:
        if c == 0x80:
            continue
        assert oracle.e4m3_encode(vals[c], mutant) == c, hex(c)
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.standard_normal(1500) * 10.0 ** rng.uniform(-3.5, 2.8, 1500),
                         (vals[finite][:-1] + np.roll(vals[finite], -1)[:-1]) / 2])
    for x in xs.astype(np.float32):
        x = float(x)
        if abs(x) >= 448.0:
            want_v = math.copysign(448.0, x)
        else:
            dist = [abs(vals[c] - x) for c in finite]
            best = min(dist)
            cands = [c for c, dd in zip(finite, dist) if dd == best]
            if len(cands) > 1:           # a tie: the even mantissa
                cands = [c for c in cands if (c & 1) == 0] or cands
            want_v = vals[cands[0]]
        got = oracle.e4m3_encode(x, mutant)
        assert vals[got] == want_v, (x, hex(got), want_v)


def pin_fp8_block_quant(mutant=0):
    """One scale per 128-row block: scale = amax / 448 (fp32), the amax
    element encodes to +-448, and every value comes back within half a step:
    |x - decode(code) * scale| <= max(2^-4 |x|, 2^-10 scale).  V's codes are
    the transpose of the same block quantised without transposing."""
    rng = np.random.default_rng(9)
    B, H, Hkv, N, d = 1, 2, 1, 200, 128
    q = (rng.standard_normal((B, H, N, d)) * 3).astype(np.float32)
    k = (rng.standard_normal((B, Hkv, N, d)) * 0.01).astype(np.float32)
    v = rng.standard_normal((B, Hkv, N, d)).astype(np.float32)
    v[0, 0, 5, 7] = 40.0
    qd = oracle.fp8_quantize(q, k, v, mutant)
    table = np.array([_e4m3_value_by_definition(c) for c in range(256)])
    for name, x, codes, sc in (("q", q.reshape(2, N, d), qd["q8"], qd["sq"]),
                               ("k", k.reshape(1, N, d), qd["k8"], qd["sk"])):
        for g in range(x.shape[0]):
            for b in range(2):
                blk = x[g, b * 128:(b + 1) * 128]
                amax = np.float32(np.abs(blk).max())
                assert sc[g, b] == np.float32(amax / np.float32(448.0)), name
                cb = codes[g, b * 128:b * 128 + blk.shape[0]]
                assert (cb & 0x7F).max() == 0x7E, name
                back = table[cb] * float(sc[g, b])
                bound = np.maximum(2.0 ** -4 * np.abs(blk), 2.0 ** -10 * float(sc[g, b]))
                assert np.all(np.abs(blk - back) <= bound + 1e-30), name
    assert qd["svmax"][0] == np.float32(40.0 / 448.0)
    plain = oracle.fp8_quantize(v.reshape(1, 1, N, d), v, v, mutant)["q8"]
    assert np.array_equal(np.swapaxes(qd["v8t"], 1, 2), plain)
    # V alone (the operand the FP8 forward quantises): the same codes and
    # scales, and the values they stand for within half a step of V
    qv = oracle.fp8_quantize_v(v, mutant)
    assert np.array_equal(qv["v8t"], qd["v8t"]) and np.array_equal(qv["sv"], qd["sv"])
    back = oracle.fp8_dequantize_v(qv, B, Hkv, N, d)
    svr = np.repeat(qv["sv"][0].astype(np.float64), 128)[:N, None]
    assert np.all(np.abs(v[0, 0] - back[0, 0]) <=
                  np.maximum(2.0 ** -4 * np.abs(v[0, 0]), 2.0 ** -10 * svr) + 1e-30)


def pin_incoherent_rotation(mutant=0):
    """The rotation of incoherent processing (reading of the FlashAttention-3
    summary's abstract): M = diag(signs) Hd / sqrt(d).  d = 2 and d = 4 against
    the textbook Hadamard matrices written out by hand; M orthogonal at
    d = 128; rotating Q and K by the same M leaves attention unchanged."""
    r2 = 1.0 / math.sqrt(2.0)
    got = oracle.incoherent_rotate(np.array([[3.0, 5.0]]), [1, -1], mutant)
    assert np.allclose(got, [[(3.0 - 5.0) * r2, (3.0 + 5.0) * r2]], rtol=0, atol=1e-14)
    h4 = 0.5 * np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], float)
    assert np.array_equal(oracle.incoherent_rotate(np.eye(4), [1, 1, 1, 1], mutant), h4)
    rng = np.random.default_rng(11)
    signs = rng.choice([-1, 1], 128)
    m = oracle.incoherent_rotate(np.eye(128), signs, mutant)
    assert np.abs(m @ m.T - np.eye(128)).max() <= 1e-12
    q, k, v = rand_qkv(1, 2, 1, 96, 128, 12)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.088)
    ro, rl = oracle.attn_fwd(oracle.incoherent_rotate(q, signs, mutant),
                             oracle.incoherent_rotate(k, signs, mutant), v, True, 0.088)
    assert np.abs(ro - o).max() <= 1e-12 and np.abs(rl - lse).max() <= 1e-12


def pin_decode_rows(mutant=0):
    """Fewer queries than keys: with the queries taken as the last Nq rows of a
    square problem, the result equals those rows of the square oracle (causal
    and not), and a library special case (torch fp64 softmax with an explicit
    bottom-right mask) agrees."""
    rng = np.random.default_rng(11)
    B, H, Hkv, Nk, d, scale = 1, 4, 2, 37, 16, 0.3
    q = rng.standard_normal((B, H, Nk, d))
    k = rng.standard_normal((B, Hkv, Nk, d))
    v = rng.standard_normal((B, Hkv, Nk, d))
    for causal in (False, True):
        ro, rl = oracle.attn_fwd(q, k, v, causal, scale)
        for nq in (1, 5, Nk):
            o, l = oracle.attn_fwd_decode(q[:, :, Nk - nq:], k, v, causal, scale, mutant)
            assert np.allclose(o, ro[:, :, Nk - nq:], rtol=1e-12, atol=1e-12), (causal, nq)
            assert np.allclose(l, rl[:, :, Nk - nq:], rtol=1e-12, atol=1e-12), (causal, nq)
    nq = 3
    qt = torch.as_tensor(q[:, :, Nk - nq:])
    kt = torch.as_tensor(k).repeat_interleave(H // Hkv, dim=1)
    vt = torch.as_tensor(v).repeat_interleave(H // Hkv, dim=1)
    s = qt @ kt.transpose(-1, -2) * scale
    r = torch.arange(nq)[:, None] + (Nk - nq)
    s = s.masked_fill(torch.arange(Nk)[None, :] > r, float("-inf"))
    want = torch.softmax(s, -1) @ vt
    o, _ = oracle.attn_fwd_decode(q[:, :, Nk - nq:], k, v, True, scale, mutant)
    assert np.allclose(o, want.numpy(), rtol=1e-12, atol=1e-12)


def pin_sliding_window(mutant=0):
    """Causal sliding window (query i sees keys i - W < j <= i): a window of N
    or more is the causal result (forward and gradients); W = 1 gives
    O_i = V_i and LSE_i = scale q_i.k_i exactly; a library special case (torch
    fp64 softmax with an explicit band mask, and its autograd) agrees."""
    rng = np.random.default_rng(12)
    B, H, Hkv, N, d, scale = 1, 4, 2, 29, 8, 0.35
    q, k, v, do = rand_qkv(B, H, Hkv, N, d, 12, dout=True)
    ro, rl = oracle.attn_fwd(q, k, v, True, scale)
    o, l = oracle.attn_fwd_window(q, k, v, N + 3, scale, mutant)
    assert np.allclose(o, ro, rtol=1e-12, atol=1e-12) and np.allclose(l, rl, rtol=1e-12, atol=1e-12)
    g_ref = oracle.attn_bwd(q, k, v, do, True, scale)
    g_w = oracle.attn_bwd_window(q, k, v, do, N, scale, mutant)
    for a, b in zip(g_ref, g_w):
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    o1, l1 = oracle.attn_fwd_window(q, k, v, 1, scale, mutant)
    G = H // Hkv
    vv = np.repeat(v, G, axis=1)
    kk = np.repeat(k, G, axis=1)
    assert np.allclose(o1, vv, rtol=1e-12, atol=1e-12)
    assert np.allclose(l1, scale * np.einsum("bhnd,bhnd->bhn", q, kk), rtol=1e-12, atol=1e-12)
    W = 5
    qt, kt, vt, dot = (torch.tensor(x, requires_grad=True) for x in (q, k, v, do))
    ke, ve = kt.repeat_interleave(G, dim=1), vt.repeat_interleave(G, dim=1)
    s = qt @ ke.transpose(-1, -2) * scale
    i_ = torch.arange(N)[:, None]
    j_ = torch.arange(N)[None, :]
    s = s.masked_fill((j_ > i_) | (i_ - j_ >= W), float("-inf"))
    out = torch.softmax(s, -1) @ ve
    (out * dot.detach()).sum().backward()
    ow, _ = oracle.attn_fwd_window(q, k, v, W, scale, mutant)
    assert np.allclose(ow, out.detach().numpy(), rtol=1e-12, atol=1e-12)
    gq, gk, gv, _ = oracle.attn_bwd_window(q, k, v, do, W, scale, mutant)
    assert np.allclose(gq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(gk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(gv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)


def pin_window_slice(mutant=0):
    """Windowed attention of a row depends only on the W positions ending at
    it: the oracle on the slice [s, e) of the sequence reproduces the forward
    and dQ of rows i >= s + W - 1 and dK, dV of keys j in [s + W - 1, e - W + 1)
    of the whole sequence (the reduction the full-size GPU test relies on)."""
    B, H, Hkv, N, d, scale, W = 1, 2, 1, 61, 8, 0.4, 9
    q, k, v, do = rand_qkv(B, H, Hkv, N, d, 13, dout=True)
    fo, fl = oracle.attn_fwd_window(q, k, v, W, scale, mutant)
    fq, fk, fv, _ = oracle.attn_bwd_window(q, k, v, do, W, scale, mutant)
    s, e = 17, 49
    sl = lambda x: np.ascontiguousarray(x[:, :, s:e])
    so, sl_ = oracle.attn_fwd_window(sl(q), sl(k), sl(v), W, scale, mutant)
    sq, sk, sv, _ = oracle.attn_bwd_window(sl(q), sl(k), sl(v), sl(do), W, scale, mutant)
    r0, k1 = W - 1, (e - s) - W + 1
    close = lambda a, b: np.allclose(a, b, rtol=1e-12, atol=1e-12)
    assert close(so[:, :, r0:], fo[:, :, s + r0:e]) and close(sl_[:, :, r0:], fl[:, :, s + r0:e])
    assert close(sq[:, :, r0:], fq[:, :, s + r0:e])
    assert close(sk[:, :, r0:k1], fk[:, :, s + r0:s + k1])
    assert close(sv[:, :, r0:k1], fv[:, :, s + r0:s + k1])
    # The rows before s + W - 1 do change (their windows lose keys): the
    # slice is exact only where the statement says.
    assert not close(so[:, :, 0], fo[:, :, s])


def pin_varlen(mutant=0):
    """Packed variable-length batches: with equal lengths the packed result is
    the dense batched one (forward and gradients, both masks); with ragged
    lengths (an empty and a one-row sequence among them) a torch fp64
    softmax over the whole packed row with a block-diagonal (and causal) mask,
    and its autograd, agree."""
    close = lambda a, b: np.allclose(a, b, rtol=1e-10, atol=1e-12)
    B, H, Hkv, N, d, scale = 3, 4, 2, 13, 8, 0.3
    q, k, v, do = rand_qkv(B, H, Hkv, N, d, 14, dout=True)
    pack = lambda x: np.ascontiguousarray(
        x.transpose(1, 0, *range(2, x.ndim)).reshape(x.shape[1], B * N, *x.shape[3:]))
    cu = np.arange(B + 1) * N
    for causal in (False, True):
        o, l = oracle.attn_fwd(q, k, v, causal, scale)
        ov, lv = oracle.attn_fwd_varlen(pack(q), pack(k), pack(v), cu, causal, scale, mutant)
        assert close(ov, pack(o)) and close(lv, pack(l[..., None])[..., 0])
        g = oracle.attn_bwd(q, k, v, do, causal, scale)
        gv = oracle.attn_bwd_varlen(pack(q), pack(k), pack(v), pack(do), cu, causal, scale, mutant)
        for a_, b_ in zip(gv[:3], g[:3]):
            assert close(a_, pack(b_))
    lens = [5, 0, 1, 17, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, G = int(cu[-1]), H // Hkv
    rng = np.random.default_rng(15)
    qp, dop = rng.standard_normal((H, T, d)), rng.standard_normal((H, T, d))
    kp, vp = rng.standard_normal((Hkv, T, d)), rng.standard_normal((Hkv, T, d))
    seq = np.repeat(np.arange(len(lens)), lens)
    same = torch.tensor(seq[:, None] == seq[None, :])
    for causal in (False, True):
        allowed = same & torch.tril(torch.ones(T, T, dtype=torch.bool)) if causal else same
        qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (qp, kp, vp))
        ke, ve = kt.repeat_interleave(G, dim=0), vt.repeat_interleave(G, dim=0)
        sc = (qt @ ke.transpose(-1, -2) * scale).masked_fill(~allowed, float("-inf"))
        out = torch.softmax(sc, -1) @ ve
        lse = torch.logsumexp(sc, -1)
        (out * torch.tensor(dop)).sum().backward()
        ov, lv = oracle.attn_fwd_varlen(qp, kp, vp, cu, causal, scale, mutant)
        assert close(ov, out.detach().numpy()) and close(lv, lse.detach().numpy())
        gq, gk, gv, _ = oracle.attn_bwd_varlen(qp, kp, vp, dop, cu, causal, scale, mutant)
        assert close(gq, qt.grad.numpy()) and close(gk, kt.grad.numpy())
        assert close(gv, vt.grad.numpy())


ALL_PINS = [
    pin_varlen,
    pin_sliding_window,
    pin_window_slice,
    pin_decode_rows,
    pin_e4m3_definition,
    pin_e4m3_nearest,
    pin_fp8_block_quant,
    pin_incoherent_rotation,
    pin_rows_sum_to_one, pin_torch_library, pin_online_matches_three_pass,
    pin_identical_keys, pin_one_hot, pin_causal_row0_and_single_key,
    pin_shift_invariance, pin_golden_closed_form, pin_finite_differences,
    pin_torch_autograd, pin_backward_invariants, pin_gqa_equals_repeated_mha,
    pin_row_subset,
]
