"""Pins of the fp64 oracle against things other than itself.

Every check here runs on the CPU. The oracle is compared with: a hand-derived
worked example (tests/golden), pure-Python brute force, central finite
differences, closed forms, invariants of softmax attention, torch's fp64
scaled_dot_product_attention with autograd, and the two independent statements
of the log-sum-exp merge. ``test_planted_mistakes`` then plants typical
mistakes into a copy of the oracle and checks that these pins catch each one.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_l2.json")

MASKS = [
    # (is_causal, window)
    (False, (-1, -1)),
    (True, (-1, -1)),
    (True, (0, 0)),
    (True, (2, 0)),
    (False, (1, 1)),
    (False, (-1, 1)),
    (False, (2, -1)),
]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _tiny(seed, l=7, h=2, hkv=1, d=4, n=1):
    q = _rand((n, l, h, d), seed)
    k = _rand((n, l, hkv, d), seed + 1)
    v = _rand((n, l, hkv, d), seed + 2)
    do = _rand((n, l, h, d), seed + 3)
    return q, k, v, do


# ---------------------------------------------------------------------------
# golden worked example
# ---------------------------------------------------------------------------

def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln3": math.log(3), "ln2": math.log(2), "ln4": math.log(4),
             "0.75ln3": 0.75 * math.log(3), "-0.75ln3": -0.75 * math.log(3)}
    return table[x]


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(x) for x in nested], dtype=np.float64)
    return _num(nested)


@pytest.mark.parametrize("mode", ["full", "causal"])
def test_golden_worked_example(mode):
    g = json.load(open(GOLDEN))
    q = _arr(g["inputs"]["q"])[None]
    k = _arr(g["inputs"]["k"])[None]
    v = _arr(g["inputs"]["v"])[None]
    do = _arr(g["inputs"]["dout"])[None]
    causal = mode == "causal"
    exp = g["expected"][mode]
    out, lse = oracle.attention_fwd(q, k, v, 1.0, causal)
    np.testing.assert_allclose(out[0], _arr(exp["out"]), atol=1e-14)
    np.testing.assert_allclose(lse[0], _arr(exp["lse"]), atol=1e-14)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, 1.0, causal)
    np.testing.assert_allclose(dq[0], _arr(exp["dq"]), atol=1e-14)
    np.testing.assert_allclose(dk[0], _arr(exp["dk"]), atol=1e-14)
    np.testing.assert_allclose(dv[0], _arr(exp["dv"]), atol=1e-14)


def test_golden_merge():
    g = json.load(open(GOLDEN))["expected"]["merge_row0"]
    oa_ = np.array(g["a"]["out"]).reshape(1, 1, 1, 2)
    ob_ = np.array(g["b"]["out"]).reshape(1, 1, 1, 2)
    la = np.array([_num(g["a"]["lse"])]).reshape(1, 1, 1)
    lb = np.array([_num(g["b"]["lse"])]).reshape(1, 1, 1)
    for fn in (oracle.merge_max_form, oracle.merge_sigmoid_form):
        o, l = fn(oa_, la, ob_, lb)
        np.testing.assert_allclose(o.ravel(), g["merged"]["out"], atol=1e-14)
        np.testing.assert_allclose(l.ravel(), [_num(g["merged"]["lse"])], atol=1e-14)


# ---------------------------------------------------------------------------
# brute force: scalar Python loops with math.fsum
# ---------------------------------------------------------------------------

def _bf_visible(i, j, causal, window):
    left, right = window
    if causal:
        right = 0
    if left >= 0 and j < i - left:
        return False
    if right >= 0 and j > i + right:
        return False
    return True


def _brute(q, k, v, do, scale, causal, window):
    n, l, h, d = q.shape
    hkv = k.shape[2]
    g = h // hkv
    out = np.zeros_like(q)
    lse = np.full((n, h, l), -np.inf)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(n):
        for hq in range(h):
            kv = hq // g
            for i in range(l):
                keys = [j for j in range(l) if _bf_visible(i, j, causal, window)]
                if not keys:
                    continue
                s = {j: scale * math.fsum(q[b, i, hq, c] * k[b, j, kv, c] for c in range(d))
                     for j in keys}
                m = max(s.values())
                z = math.fsum(math.exp(s[j] - m) for j in keys)
                lse[b, hq, i] = m + math.log(z)
                p = {j: math.exp(s[j] - m) / z for j in keys}
                o = [math.fsum(p[j] * v[b, j, kv, c] for j in keys) for c in range(d)]
                out[b, i, hq, :] = o
                # gradient of sum(do * out) through the softmax Jacobian:
                # d out_c / d s_j = p_j (v_jc - out_c)
                ds = {}
                for j in keys:
                    ds[j] = p[j] * math.fsum(do[b, i, hq, c] * (v[b, j, kv, c] - o[c])
                                             for c in range(d))
                for c in range(d):
                    dq[b, i, hq, c] = scale * math.fsum(ds[j] * k[b, j, kv, c] for j in keys)
                for j in keys:
                    for c in range(d):
                        dk[b, j, kv, c] += scale * ds[j] * q[b, i, hq, c]
                        dv[b, j, kv, c] += p[j] * do[b, i, hq, c]
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("causal,window", MASKS)
@pytest.mark.parametrize("h,hkv", [(2, 1), (2, 2)])
def test_brute_force(causal, window, h, hkv):
    q, k, v, do = _tiny(11, l=8, h=h, hkv=hkv, d=4)
    scale = 0.7
    out, lse = oracle.attention_fwd(q, k, v, scale, causal, window)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, scale, causal, window)
    bo, bl, bdq, bdk, bdv = _brute(q, k, v, do, scale, causal, window)
    np.testing.assert_allclose(out, bo, atol=1e-12)
    np.testing.assert_allclose(lse, bl, atol=1e-12)
    np.testing.assert_allclose(dq, bdq, atol=1e-12)
    np.testing.assert_allclose(dk, bdk, atol=1e-12)
    np.testing.assert_allclose(dv, bdv, atol=1e-12)


def test_row_subset_matches_full():
    q, k, v, _ = _tiny(5, l=40, h=2, hkv=1, d=8)
    rows = np.array([0, 3, 17, 39])
    for causal, window in MASKS:
        out, lse = oracle.attention_fwd(q, k, v, 0.5, causal, window)
        so, sl = oracle.attention_fwd(q, k, v, 0.5, causal, window, rows=rows)
        np.testing.assert_allclose(so, out[:, rows], atol=1e-13)
        np.testing.assert_allclose(sl, lse[:, :, rows], atol=1e-13)


def test_row_blocks_do_not_change_results():
    q, k, v, do = _tiny(6, l=50, h=2, hkv=2, d=8)
    for causal, window in MASKS:
        o1, l1 = oracle.attention_fwd(q, k, v, 0.4, causal, window, row_block=1024)
        o2, l2 = oracle.attention_fwd(q, k, v, 0.4, causal, window, row_block=7)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l1, l2, atol=1e-13)
        g1 = oracle.attention_bwd(do, q, k, v, o1, l1, 0.4, causal, window, row_block=1024)
        g2 = oracle.attention_bwd(do, q, k, v, o1, l1, 0.4, causal, window, row_block=7)
        for a, b in zip(g1, g2):
            np.testing.assert_allclose(a, b, atol=1e-12)


# ---------------------------------------------------------------------------
# finite differences
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,window", MASKS)
def test_finite_differences(causal, window):
    q, k, v, do = _tiny(21, l=6, h=2, hkv=1, d=3)
    scale = 0.9
    out, lse = oracle.attention_fwd(q, k, v, scale, causal, window)
    grads = oracle.attention_bwd(do, q, k, v, out, lse, scale, causal, window)

    def f(qq, kk, vv):
        o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal, window)
        return float(np.sum(do * o))

    eps = 1e-6
    for which, (arr, grad) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [q.copy(), k.copy(), v.copy()]
            minus = [q.copy(), k.copy(), v.copy()]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (f(*plus) - f(*minus)) / (2 * eps)
        err = np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(num)))
        assert err < 1e-6, (which, err)


# ---------------------------------------------------------------------------
# softmax rows, closed forms, invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,window", MASKS)
def test_softmax_rows(causal, window):
    q, k, v, _ = _tiny(31, l=9, h=2, hkv=1, d=4)
    P = oracle.attention_probs(q, k, 0.8, causal, window)
    vis = oracle.visible_mask(np.arange(9), 9, causal, window)
    assert np.all(np.abs(P.sum(-1) - 1.0) <= 1e-12)
    assert np.all(P[..., ~vis] == 0.0)
    out, _ = oracle.attention_fwd(q, k, v, 0.8, causal, window)
    np.testing.assert_allclose(out[0, :, 0], P[0, 0] @ v[0, :, 0], atol=1e-13)


def test_closed_form_single_key():
    q, k, v, _ = _tiny(41, l=1, h=2, hkv=1, d=5)
    out, lse = oracle.attention_fwd(q, k, v, 0.3, False)
    np.testing.assert_allclose(out[0, 0, 0], v[0, 0, 0], atol=1e-15)
    np.testing.assert_allclose(lse[0, :, 0], 0.3 * (q[0, 0] @ k[0, 0, 0]), atol=1e-14)


@pytest.mark.parametrize("causal,window", MASKS)
def test_closed_form_zero_query(causal, window):
    _, k, v, _ = _tiny(42, l=10, h=1, hkv=1, d=3)
    q = np.zeros((1, 10, 1, 3))
    out, lse = oracle.attention_fwd(q, k, v, 1.0, causal, window)
    vis = oracle.visible_mask(np.arange(10), 10, causal, window)
    for i in range(10):
        js = np.nonzero(vis[i])[0]
        np.testing.assert_allclose(out[0, i, 0], v[0, js, 0].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(lse[0, 0, i], math.log(len(js)), atol=1e-14)


def test_closed_form_causal_row0_and_diagonal_window():
    q, k, v, do = _tiny(43, l=8, h=2, hkv=2, d=4)
    out, lse = oracle.attention_fwd(q, k, v, 0.5, True)
    np.testing.assert_allclose(out[0, 0], v[0, 0], atol=1e-15)
    out, lse = oracle.attention_fwd(q, k, v, 0.5, True, (0, 0))
    np.testing.assert_allclose(out, v, atol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * np.einsum("ihd,ihd->hi", q[0], k[0]), atol=1e-14)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, 0.5, True, (0, 0))
    assert np.max(np.abs(dq)) < 1e-14 and np.max(np.abs(dk)) < 1e-14
    np.testing.assert_allclose(dv, do, atol=1e-15)


@pytest.mark.parametrize("causal,window", MASKS)
def test_gradient_invariants(causal, window):
    q, k, v, do = _tiny(51, l=12, h=4, hkv=2, d=5)
    out, lse = oracle.attention_fwd(q, k, v, 0.6, causal, window)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, 0.6, causal, window)
    # softmax over keys is shift invariant -> key gradients sum to zero
    assert np.max(np.abs(dk.sum(axis=1))) < 1e-12
    # every row sees >= 1 key -> column sums of P total one per row
    g = 2
    do_sum = do.reshape(1, 12, 2, g, 5).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), do_sum, atol=1e-12)


@pytest.mark.parametrize("causal,window", MASKS)
def test_key_shift_invariance(causal, window):
    q, k, v, _ = _tiny(52, l=9, h=2, hkv=1, d=4)
    c = np.array([0.3, -1.2, 0.7, 2.0])
    out, lse = oracle.attention_fwd(q, k, v, 0.5, causal, window)
    out2, lse2 = oracle.attention_fwd(q, k + c, v, 0.5, causal, window)
    np.testing.assert_allclose(out2, out, atol=1e-12)
    shift = 0.5 * np.einsum("nlhd,d->nhl", q, c)
    np.testing.assert_allclose(lse2, lse + shift, atol=1e-12)


@pytest.mark.parametrize("causal,window", MASKS)
def test_gqa_equals_repeated_mha(causal, window):
    q, k, v, do = _tiny(53, l=10, h=6, hkv=2, d=4)
    g = 3
    krep = np.repeat(k, g, axis=2)
    vrep = np.repeat(v, g, axis=2)
    out, lse = oracle.attention_fwd(q, k, v, 0.5, causal, window)
    out_r, lse_r = oracle.attention_fwd(q, krep, vrep, 0.5, causal, window)
    np.testing.assert_allclose(out, out_r, atol=1e-14)
    np.testing.assert_allclose(lse, lse_r, atol=1e-14)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, 0.5, causal, window)
    dq_r, dk_r, dv_r = oracle.attention_bwd(do, q, krep, vrep, out, lse, 0.5, causal, window)
    np.testing.assert_allclose(dq, dq_r, atol=1e-13)
    np.testing.assert_allclose(dk, dk_r.reshape(1, 10, 2, g, 4).sum(3), atol=1e-13)
    np.testing.assert_allclose(dv, dv_r.reshape(1, 10, 2, g, 4).sum(3), atol=1e-13)


def test_empty_rows_and_keys():
    q, k, v, do = _tiny(54, l=5, h=1, hkv=1, d=3)
    out, lse = oracle.attention_fwd(q, k[:, :0], v[:, :0], 1.0, False)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
    dq, dk, dv = oracle.attention_bwd(do, q, k[:, :0], v[:, :0], out, lse, 1.0, False)
    assert np.all(dq == 0) and dk.shape == (1, 0, 1, 3)


# ---------------------------------------------------------------------------
# torch fp64 library special case
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal,window", MASKS)
def test_torch_sdpa_fp64(causal, window):
    torch = pytest.importorskip("torch")
    q, k, v, do = _tiny(61, l=16, h=4, hkv=2, d=8, n=2)
    scale = 1 / math.sqrt(8)
    out, lse = oracle.attention_fwd(q, k, v, scale, causal, window)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, out, lse, scale, causal, window)
    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_()
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_()
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_()
    mask = torch.tensor(oracle.visible_mask(np.arange(16), 16, causal, window))
    kr = tk.repeat_interleave(2, dim=1)
    vr = tv.repeat_interleave(2, dim=1)
    to = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, attn_mask=mask, scale=scale)
    to.backward(torch.tensor(do).permute(0, 2, 1, 3))
    np.testing.assert_allclose(to.detach().permute(0, 2, 1, 3).numpy(), out, atol=1e-10)
    np.testing.assert_allclose(tq.grad.permute(0, 2, 1, 3).numpy(), dq, atol=1e-10)
    np.testing.assert_allclose(tk.grad.permute(0, 2, 1, 3).numpy(), dk, atol=1e-10)
    np.testing.assert_allclose(tv.grad.permute(0, 2, 1, 3).numpy(), dv, atol=1e-10)
    s = scale * torch.einsum("bhid,bhjd->bhij", tq.detach(), kr.detach())
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(torch.logsumexp(s, dim=-1).numpy(), lse, atol=1e-10)


# ---------------------------------------------------------------------------
# merge and ring replay
# ---------------------------------------------------------------------------

def test_merge_reproduces_unchunked_attention():
    rng = np.random.default_rng(71)
    q, k, v, _ = _tiny(72, l=20, h=2, hkv=1, d=4)
    ref_o, ref_l = oracle.attention_fwd(q, k, v, 0.5, False)
    for trial in range(10):
        perm = rng.permutation(20)
        cuts = np.sort(rng.choice(np.arange(0, 21), size=3, replace=True))
        parts = np.split(perm, cuts)          # may contain empty parts
        o_acc = np.zeros_like(q)
        l_acc = np.full((1, 2, 20), -np.inf)
        for part in parts:
            ob, lb = oracle.attention_fwd(q, k[:, part], v[:, part], 0.5, False)
            fn = oracle.merge_max_form if trial % 2 else oracle.merge_sigmoid_form
            o_acc, l_acc = fn(o_acc, l_acc, ob, lb)
        np.testing.assert_allclose(o_acc, ref_o, atol=1e-12)
        np.testing.assert_allclose(l_acc, ref_l, atol=1e-12)


def test_merge_algebra():
    rng = np.random.default_rng(73)
    shape_o, shape_l = (2, 6, 3, 4), (2, 3, 6)
    os_ = [rng.standard_normal(shape_o) for _ in range(3)]
    ls = [rng.standard_normal(shape_l) * 3 for _ in range(3)]
    ls[1][0, 0, :2] = -np.inf          # some dead rows
    ls[2][1, 2, 3] = -np.inf
    ls[1][1, 2, 3] = -np.inf           # both dead at one row of (1, 2)
    m = oracle.merge_max_form
    # commutative
    a = m(os_[0], ls[0], os_[1], ls[1])
    b = m(os_[1], ls[1], os_[0], ls[0])
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)
    # associative
    x = m(*m(os_[0], ls[0], os_[1], ls[1]), os_[2], ls[2])
    y = m(os_[0], ls[0], *m(os_[1], ls[1], os_[2], ls[2]))
    np.testing.assert_allclose(x[0], y[0], atol=1e-12)
    np.testing.assert_allclose(x[1], y[1], atol=1e-12)
    # identity element (., -inf), exactly
    dead = np.full(shape_l, -np.inf)
    z = m(os_[0], ls[0], os_[1], dead)
    assert np.array_equal(z[0], os_[0]) and np.array_equal(z[1], ls[0])
    z = m(np.zeros(shape_o), dead, os_[1], ls[1])
    live = np.isfinite(ls[1])
    assert np.array_equal(z[0][np.transpose(live, (0, 2, 1))], os_[1][np.transpose(live, (0, 2, 1))])
    # self merge doubles the weight
    z = m(os_[0], ls[0], os_[0], ls[0])
    np.testing.assert_allclose(z[0], os_[0], atol=1e-13)
    np.testing.assert_allclose(z[1], ls[0] + math.log(2), atol=1e-13)
    # the two statements of the merge agree
    for i in range(3):
        for j in range(3):
            p = oracle.merge_max_form(os_[i], ls[i], os_[j], ls[j])
            s = oracle.merge_sigmoid_form(os_[i], ls[i], os_[j], ls[j])
            np.testing.assert_allclose(p[0], s[0], atol=1e-12)
            np.testing.assert_allclose(p[1], s[1], atol=1e-12)


def test_ring_schedule_counts():
    s = oracle.ring_chunk_schedule(8, True)
    kinds = [kind for steps in s for (_t, _j, kind) in steps]
    assert kinds.count("causal") == 8 and kinds.count("full") == 28 and kinds.count("skip") == 28
    for i, steps in enumerate(s):
        assert steps[0] == (0, i, "causal")          # step 0 is the diagonal
        assert sorted(j for _t, j, _k in steps) == list(range(8))


@pytest.mark.parametrize("causal", [True, False])
def test_ring_replay_matches_single_call(causal):
    q, k, v, do = _tiny(81, l=24, h=2, hkv=2, d=4)
    out, lse = oracle.attention_fwd(q, k, v, 0.5, causal)
    ro, rl = oracle.ring_fwd_replay(q, k, v, 0.5, 4, causal)
    np.testing.assert_allclose(ro, out, atol=1e-12)
    np.testing.assert_allclose(rl, lse, atol=1e-12)
    g = oracle.attention_bwd(do, q, k, v, out, lse, 0.5, causal)
    rg = oracle.ring_bwd_replay(do, q, k, v, out, lse, 0.5, 4, causal)
    for a, b in zip(g, rg):
        np.testing.assert_allclose(b, a, atol=1e-12)


def test_flop_accounting():
    f, b = oracle.algorithmic_flops(1, 32, 8192, 8192, 128, True)
    assert f == 4 * 32 * 8192 ** 2 * 128 / 2 and b == 2.5 * f
    assert oracle.visible_pairs(32768, 32768, True, (1024, 0)) == 33062400
    assert oracle.visible_pairs(10, 10, True) == 55


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by the pins above
# ---------------------------------------------------------------------------

MUTATIONS = {
    "dropped_scale_fwd": ("s = softmax_scale * (q[b, idx, hq, :]", "s = (q[b, idx, hq, :]"),
    "wrong_gqa_map": ("kv = hq // g\n                s = softmax_scale * (q[b, idx",
                      "kv = hq % hkv\n                s = softmax_scale * (q[b, idx"),
    "window_off_by_one": ("vis &= j >= i - left", "vis &= j > i - left"),
    "d_from_dp": ("D = np.sum(do * out[b, r0:r1, hq, :], axis=1)", "D = np.sum(dp, axis=1)"),
    "dk_transposed_operand": ("(ds.T @ q[b, r0:r1, hq, :])", "(ds.T @ do)"),
    "ds_sign": ("ds = p * (dp - D[:, None])", "ds = p * (D[:, None] - dp)"),
    "merge_weight_swap": ("o = out_a * _rows_view(wa) + out_b * _rows_view(wb)",
                          "o = out_a * _rows_view(wb) + out_b * _rows_view(wa)"),
    "lse_without_max": ("row_lse = np.where(any_vis, m + np.log(ssum), NEG_INF)",
                        "row_lse = np.where(any_vis, np.log(ssum), NEG_INF)"),
    "key_offset_sign": ("j = np.arange(lk, dtype=np.int64)[None, :] + int(key_offset)",
                        "j = np.arange(lk, dtype=np.int64)[None, :] - int(key_offset)"),
    "top_left_alignment": ("return lq - lk if key_offset is None else int(key_offset)",
                           "return 0 if key_offset is None else int(key_offset)"),
    "key_band_offset_sign": ("k0 = 0 if left < 0 else min(lk, max(0, r0 - left - key_offset))",
                             "k0 = 0 if left < 0 else min(lk, max(0, r0 - left + key_offset))"),
}


def _mutant(name):
    import types
    src = open(oa.__file__).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, name
    mod = types.ModuleType("oracle_mutant_" + name)
    exec(compile(src.replace(old, new), "mutant", "exec"), mod.__dict__)
    return mod


def _pins_pass(mod):
    """Run a subset of the pins above against module ``mod``."""
    try:
        g = json.load(open(GOLDEN))
        q = _arr(g["inputs"]["q"])[None]
        k = _arr(g["inputs"]["k"])[None]
        v = _arr(g["inputs"]["v"])[None]
        do = _arr(g["inputs"]["dout"])[None]
        for mode in ("full", "causal"):
            exp = g["expected"][mode]
            out, lse = mod.attention_fwd(q, k, v, 1.0, mode == "causal")
            grads = mod.attention_bwd(do, q, k, v, out, lse, 1.0, mode == "causal")
            for got, key in zip((out, lse) + tuple(grads), ("out", "lse", "dq", "dk", "dv")):
                np.testing.assert_allclose(got[0], _arr(exp[key]), atol=1e-12)
        gm = g["expected"]["merge_row0"]
        o, l = mod.merge_max_form(np.array(gm["a"]["out"]).reshape(1, 1, 1, 2),
                                  np.array([[[_num(gm["a"]["lse"])]]]),
                                  np.array(gm["b"]["out"]).reshape(1, 1, 1, 2),
                                  np.array([[[_num(gm["b"]["lse"])]]]))
        np.testing.assert_allclose(o.ravel(), gm["merged"]["out"], atol=1e-12)
        for causal, window in MASKS:
            q, k, v, do = _tiny(11, l=8, h=4, hkv=2, d=4)
            out, lse = mod.attention_fwd(q, k, v, 0.7, causal, window)
            grads = mod.attention_bwd(do, q, k, v, out, lse, 0.7, causal, window)
            bo, bl, bdq, bdk, bdv = _brute(q, k, v, do, 0.7, causal, window)
            for a, b in zip((out, lse) + tuple(grads), (bo, bl, bdq, bdk, bdv)):
                np.testing.assert_allclose(a, b, atol=1e-12)
        # unequal lengths: explicit offsets and the default (bottom-right) alignment
        q = _rand((1, 6, 2, 4), 71)
        k = _rand((1, 9, 1, 4), 72)
        v = _rand((1, 9, 1, 4), 73)
        do = _rand((1, 6, 2, 4), 74)
        for causal, window in MASKS:
            for off in (-6, -2, None, 3):
                out, lse = mod.attention_fwd(q, k, v, 0.6, causal, window, key_offset=off)
                grads = mod.attention_bwd(do, q, k, v, out, lse, 0.6, causal, window, key_offset=off)
                ref = _brute_offset(q, k, v, do, 0.6, causal, window, 6 - 9 if off is None else off)
                for a, b in zip((out, lse) + tuple(grads), ref):
                    np.testing.assert_allclose(a, b, atol=1e-12)
    except AssertionError:
        return False
    return True


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass(oa)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes(name):
    assert not _pins_pass(_mutant(name)), f"mutation {name} went unnoticed"


# ---------------------------------------------------------------------------
# key positions offset from query positions (lq != lk, ring chunk pairs)
# ---------------------------------------------------------------------------

def _brute_offset(q, k, v, do, scale, causal, window, off):
    """Scalar loops with key j at query position j + off (the reading of the
    module doc), any lq and lk."""
    n, lq, h, d = q.shape
    lk, hkv = k.shape[1], k.shape[2]
    g = h // hkv
    out = np.zeros_like(q)
    lse = np.full((n, h, lq), -np.inf)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(n):
        for hq in range(h):
            kv = hq // g
            for i in range(lq):
                keys = [j for j in range(lk) if _bf_visible(i, j + off, causal, window)]
                if not keys:
                    continue
                s = {j: scale * math.fsum(q[b, i, hq, c] * k[b, j, kv, c] for c in range(d)) for j in keys}
                m = max(s.values())
                z = math.fsum(math.exp(s[j] - m) for j in keys)
                lse[b, hq, i] = m + math.log(z)
                p = {j: math.exp(s[j] - m) / z for j in keys}
                o = [math.fsum(p[j] * v[b, j, kv, c] for j in keys) for c in range(d)]
                out[b, i, hq, :] = o
                ds = {j: p[j] * math.fsum(do[b, i, hq, c] * (v[b, j, kv, c] - o[c]) for c in range(d))
                      for j in keys}
                for c in range(d):
                    dq[b, i, hq, c] = scale * math.fsum(ds[j] * k[b, j, kv, c] for j in keys)
                for j in keys:
                    for c in range(d):
                        dk[b, j, kv, c] += scale * ds[j] * q[b, i, hq, c]
                        dv[b, j, kv, c] += p[j] * do[b, i, hq, c]
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("causal,window", MASKS)
@pytest.mark.parametrize("off", [-6, -2, 0, 3])
def test_brute_force_key_offset(causal, window, off):
    q = _rand((1, 6, 2, 4), 71)
    k = _rand((1, 9, 1, 4), 72)
    v = _rand((1, 9, 1, 4), 73)
    do = _rand((1, 6, 2, 4), 74)
    out, lse = oracle.attention_fwd(q, k, v, 0.6, causal, window, key_offset=off)
    grads = oracle.attention_bwd(do, q, k, v, out, lse, 0.6, causal, window, key_offset=off)
    ref = _brute_offset(q, k, v, do, 0.6, causal, window, off)
    for got, want in zip((out, lse) + tuple(grads), ref):
        np.testing.assert_allclose(got, want, atol=1e-12)


@pytest.mark.parametrize("causal,window", MASKS)
def test_bottom_right_is_the_suffix_of_the_square(causal, window):
    """Default alignment for lq < lk: the last query row sees up to the last key, so the lq
    rows are exactly the last lq rows of the square computation over all lk queries."""
    lk, lq = 11, 4
    q, k, v, do = _tiny(81, l=lk, h=2, hkv=1, d=4)
    full_o, full_l = oracle.attention_fwd(q, k, v, 0.8, causal, window)
    o, l_ = oracle.attention_fwd(q[:, lk - lq:], k, v, 0.8, causal, window)
    np.testing.assert_allclose(o, full_o[:, lk - lq:], atol=1e-13)
    np.testing.assert_allclose(l_, full_l[:, :, lk - lq:], atol=1e-13)
    # dq of those rows does not depend on the other query rows
    do_sfx = do[:, lk - lq:]
    dq, _, _ = oracle.attention_bwd(do_sfx, q[:, lk - lq:], k, v, o, l_, 0.8, causal, window)
    do_full = np.zeros_like(do)
    do_full[:, lk - lq:] = do_sfx
    fdq, _, _ = oracle.attention_bwd(do_full, q, k, v, full_o, full_l, 0.8, causal, window)
    np.testing.assert_allclose(dq, fdq[:, lk - lq:], atol=1e-13)


@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (True, (5, 0)), (False, (4, 3))])
def test_key_chunks_with_offsets_merge_to_the_whole(causal, window):
    """Rows [a, b) of attention over all keys = the merge, over key chunks [c0, c1), of
    attention of those rows against the chunk placed at offset c0 - a."""
    l = 16
    q, k, v, _ = _tiny(91, l=l, h=2, hkv=2, d=4)
    full_o, full_l = oracle.attention_fwd(q, k, v, 0.7, causal, window)
    a, b = 5, 12
    acc_o = np.zeros((1, b - a, 2, 4))
    acc_l = np.full((1, 2, b - a), -np.inf)
    for c0, c1 in ((0, 3), (3, 8), (8, 13), (13, 16)):
        o_, l_ = oracle.attention_fwd(q[:, a:b], k[:, c0:c1], v[:, c0:c1], 0.7, causal, window,
                                      key_offset=c0 - a)
        acc_o, acc_l = oracle.merge_max_form(acc_o, acc_l, o_, l_)
    np.testing.assert_allclose(acc_o, full_o[:, a:b], atol=1e-12)
    np.testing.assert_allclose(acc_l, full_l[:, :, a:b], atol=1e-12)


@pytest.mark.parametrize("causal,window", [(True, (5, 0)), (False, (3, 2)), (True, (0, 0))])
def test_windowed_ring_replay_matches_single_call(causal, window):
    q, k, v, do = _tiny(95, l=24, h=2, hkv=1, d=4)
    o, l_ = oracle.ring_fwd_replay(q, k, v, 0.5, 4, causal, window)
    so, sl = oracle.attention_fwd(q, k, v, 0.5, causal, window)
    np.testing.assert_allclose(o, so, atol=1e-12)
    np.testing.assert_allclose(l_, sl, atol=1e-12)
    g = oracle.ring_bwd_replay(do, q, k, v, so, sl, 0.5, 4, causal, window)
    sg = oracle.attention_bwd(do, q, k, v, so, sl, 0.5, causal, window)
    for a_, b_ in zip(g, sg):
        np.testing.assert_allclose(a_, b_, atol=1e-12)


def test_finite_differences_unequal_lengths():
    q = _rand((1, 4, 2, 3), 101)
    k = _rand((1, 7, 1, 3), 102)
    v = _rand((1, 7, 1, 3), 103)
    do = _rand((1, 4, 2, 3), 104)
    out, lse = oracle.attention_fwd(q, k, v, 0.9, True, (2, 0))
    grads = oracle.attention_bwd(do, q, k, v, out, lse, 0.9, True, (2, 0))

    def f(qq, kk, vv):
        return float(np.sum(do * oracle.attention_fwd(qq, kk, vv, 0.9, True, (2, 0))[0]))

    eps = 1e-6
    for which, (arr, grad) in enumerate(zip((q, k, v), grads)):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [q.copy(), k.copy(), v.copy()]
            minus = [q.copy(), k.copy(), v.copy()]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (f(*plus) - f(*minus)) / (2 * eps)
        assert np.max(np.abs(num - grad)) / max(1.0, np.max(np.abs(num))) < 1e-6, which
