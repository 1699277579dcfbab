"""Context-parallel attention: the schedule, the argument checks (no launch),
and the chunk-pair decomposition of causal attention checked against the
oracle on the CPU.

The pages say only that context parallelism splits the sequence across
ranks and that attention still needs the earlier tokens' K and V from the
other ranks (Megatron Core guide, parallelism table and the section on
proving semantics unchanged).  The reading taken: 2 cp chunks, rank r owns
chunks r and 2 cp - 1 - r, ring steps pass K/V chunks, partials merged by
log-sum-exp.
"""
import numpy as np
import pytest

import oracle.layer as O
from megatron_transformer_layer_gb300 import _lib as L


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8])
def test_schedule_covers_every_causal_chunk_pair_once(cp):
    C = 2 * cp
    seen = {}
    for r in range(cp):
        for t in range(cp):
            for i, j in L.mc_cp_schedule(cp, r, t):
                assert (i, j) not in seen, (i, j)
                seen[(i, j)] = (r, t)
                # rank r owns query chunk i; the K/V chunk j belongs to the
                # rank whose K/V r holds in step t
                assert i in (r, C - 1 - r)
                src = (r - t) % cp
                assert j in (src, C - 1 - src)
                assert j <= i
    assert set(seen) == {(i, j) for i in range(C) for j in range(i + 1)}


@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_schedule_balances_causal_work(cp):
    """Every rank computes 2 cp - 1 full chunk pairs and 2 diagonal (half)
    ones: the same causal work."""
    for r in range(cp):
        pairs = [p for t in range(cp) for p in L.mc_cp_schedule(cp, r, t)]
        diag = sum(1 for i, j in pairs if i == j)
        assert diag == 2 and len(pairs) == 2 * cp + 1


def test_schedule_rejects_bad_arguments():
    for args in [(0, 0, 0), (2, 2, 0), (2, 0, 2), (2, -1, 0)]:
        with pytest.raises(ValueError):
            L.mc_cp_schedule(*args)


def test_workspace_bytes():
    """Running fp32 sums for the whole sequence ([b, s, 3a]) plus the bf16
    dS^T tiles of one launch: up to one chunk pair per rank, [b, H, c/128,
    c/128] x 128 x 128 each.  The size does not grow with the number of CP
    partitions."""
    b, s, H, d, cp = 2, 2048, 4, 128, 4
    c, a = s // (2 * cp), H * d
    tiles = cp * b * H * (c // 128) ** 2 * 128 * 128 * 2
    assert L.mc_attention_cp_workspace_bytes(b, s, H, d, cp) == b * s * 3 * a * 4 + tiles
    sizes = [L.mc_attention_cp_workspace_bytes(1, 8192, 8, 128, k) for k in (1, 2, 4, 8)]
    assert sizes == sorted(sizes, reverse=True)
    assert L.mc_attention_cp_workspace_bytes(b, 2048 + 128, H, d, cp) == 0  # chunk not whole tiles
    assert L.mc_attention_cp_workspace_bytes(b, s, H, 96, cp) == 0
    assert L.mc_attention_cp_workspace_bytes(b, s, H, d, 0) == 0


def test_cp_entry_points_reject_bad_arguments_before_launch():
    fake = 1 << 20  # 16-byte aligned, never dereferenced: every case fails on the host
    ws = L.mc_attention_cp_workspace_bytes(1, 1024, 2, 128, 2)
    f = L.lib().mc_attention_forward_cp
    assert f(fake, fake, fake, 1, 1000, 2, 128, 2, fake, ws, None, None) == L.MC_ERR_SHAPE
    assert f(fake, fake, fake, 1, 1024, 2, 128, 0, fake, ws, None, None) == L.MC_ERR_SHAPE
    assert f(fake, fake, fake, 1, 1024, 2, 80, 2, fake, ws, None, None) == L.MC_ERR_UNSUPPORTED
    assert f(None, fake, fake, 1, 1024, 2, 128, 2, fake, ws, None, None) == L.MC_ERR_NULLPTR
    assert f(fake + 4, fake, fake, 1, 1024, 2, 128, 2, fake, ws, None, None) == L.MC_ERR_ALIGN
    assert f(fake, fake, fake, 1, 1024, 2, 128, 2, fake, ws - 1, None, None) == L.MC_ERR_WORKSPACE
    g = L.lib().mc_attention_backward_cp
    assert g(fake, fake, fake, fake, fake, fake, 1, 1024, 2, 128, 2, fake, ws - 1, None,
             None) == L.MC_ERR_WORKSPACE
    assert g(fake, fake, fake, None, fake, fake, 1, 1024, 2, 128, 2, fake, ws, None,
             None) == L.MC_ERR_NULLPTR


def _partial(q, k, v, q0, k0, causal):
    """Softmax attention of rows q (absolute positions q0..) over keys k
    (absolute positions k0..), causal mask inside; returns (O, lse)."""
    sc = (q @ k.T) / np.sqrt(q.shape[1])
    if causal:
        rows = np.arange(q.shape[0])[:, None] + q0
        cols = np.arange(k.shape[0])[None, :] + k0
        sc = np.where(cols <= rows, sc, -np.inf)
    m = sc.max(axis=1, keepdims=True)
    e = np.exp(sc - m)
    l = e.sum(axis=1, keepdims=True)
    return (e / l) @ v, (m + np.log(l))[:, 0]


@pytest.mark.parametrize("cp", [1, 2, 3])
def test_chunk_pair_partials_merge_to_causal_attention(cp):
    """The decomposition the CP path computes: merging the chunk-pair
    partials of each query chunk with the log-sum-exp rule gives the oracle's
    causal attention (and its LSE)."""
    rng = np.random.default_rng(3)
    C, c, d = 2 * cp, 8, 16
    s = C * c
    q, k, v = (rng.standard_normal((s, d)) * 1.5 for _ in range(3))
    o_ref, lse_ref = O.causal_attention_forward(q, k, v)
    o = np.empty_like(o_ref)
    lse = np.empty_like(lse_ref)
    parts = {}
    for r in range(cp):
        for t in range(cp):
            for i, j in L.mc_cp_schedule(cp, r, t):
                qs, ks = slice(i * c, (i + 1) * c), slice(j * c, (j + 1) * c)
                parts[(i, j)] = _partial(q[qs], k[ks], v[ks], i * c, j * c, i == j)
    for i in range(C):
        ls = np.stack([parts[(i, j)][1] for j in range(i + 1)])      # [pairs, c]
        l = np.log(np.exp(ls - ls.max(axis=0)).sum(axis=0)) + ls.max(axis=0)
        w = np.exp(ls - l)                                            # weights sum to 1
        o[i * c:(i + 1) * c] = sum(w[j][:, None] * parts[(i, j)][0] for j in range(i + 1))
        lse[i * c:(i + 1) * c] = l
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


MERGE, FINAL = 1, 2


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8, 17, 40])
def test_launch_plan_covers_the_schedule_without_conflicts(cp):
    """The plan the CP entry points launch: every pair j <= i exactly once;
    no launch holds two pairs of one query chunk or of one key chunk (each
    would touch a running sum twice) nor more than 16 pairs; each rank's
    pairs in the order of its ring steps."""
    plan = L.mc_cp_launch_plan(cp)
    C = 2 * cp
    assert sorted((i, j) for _, i, j, _, _ in plan) == [(i, j) for i in range(C) for j in range(i + 1)]
    launches = [entry[0] for entry in plan]
    assert launches == sorted(launches) and launches[0] == 0
    assert sorted(set(launches)) == list(range(launches[-1] + 1))
    by_launch = {}
    for l, i, j, _, _ in plan:
        by_launch.setdefault(l, []).append((i, j))
    for pairs in by_launch.values():
        qs, ks = [i for i, _ in pairs], [j for _, j in pairs]
        assert len(set(qs)) == len(qs) and len(set(ks)) == len(ks) and len(pairs) <= 16
    for r in range(cp):
        mine = [(i, j) for _, i, j, _, _ in plan if i in (r, C - 1 - r)]
        assert mine == [p for t in range(cp) for p in L.mc_cp_schedule(cp, r, t)]


@pytest.mark.parametrize("cp", [1, 2, 3, 4, 8, 17])
def test_launch_plan_accumulation_modes(cp):
    """A chunk's first pair writes its running sum, the later ones add to
    it, its last writes the result: query chunk i has i + 1 pairs, key chunk
    j has 2 cp - j."""
    plan = L.mc_cp_launch_plan(cp)
    C = 2 * cp
    for chunk in range(C):
        for pos, mpos, n in ((1, 3, chunk + 1), (2, 4, C - chunk)):
            modes = [e[mpos] for e in plan if e[pos] == chunk]
            assert len(modes) == n
            want = [FINAL] if n == 1 else [0] + [MERGE] * (n - 2) + [MERGE | FINAL]
            assert modes == want


def test_launch_plan_limits():
    assert len(L.mc_cp_launch_plan(256)) == 256 * 513
    for bad in (0, 257, -1):
        with pytest.raises(ValueError):
            L.mc_cp_launch_plan(bad)
    buf = (L.ctypes.c_int32 * 50)()
    assert L.lib().mc_cp_launch_plan(2, buf, 9) == L.MC_ERR_WORKSPACE
    assert L.lib().mc_cp_launch_plan(2, None, 10) == L.MC_ERR_ARGUMENT
    assert L.lib().mc_cp_launch_plan(2, buf, 10) == 10
    # 257 parts is beyond the plan's fixed arrays: the entry points refuse it
    assert L.mc_attention_cp_workspace_bytes(1, 256 * 257, 1, 128, 257) == 0


@pytest.mark.parametrize("cp", [1, 2, 3])
def test_running_sums_in_launch_order_give_causal_attention(cp):
    """What the context-parallel kernels compute, walked in the plan's launch
    order with its modes: each pair's O and log-sum-exp (log2 units) merged
    into its query chunk's running ones as the forward epilogue does, and
    each pair's dQ, dK, dV (from the merged LSE and delta) added to running
    sums, a chunk's last pair writing the result.  fp64: equal to the
    oracle's causal attention forward and backward to 1e-12."""
    rng = np.random.default_rng(4)
    C, c, d = 2 * cp, 8, 16
    s = C * c
    q, k, v, do = (rng.standard_normal((s, d)) * 1.5 for _ in range(4))
    o_ref, lse_ref = O.causal_attention_forward(q, k, v)
    dq_ref, dk_ref, dv_ref = O.causal_attention_backward(q, k, v, o_ref, lse_ref, do)
    plan = L.mc_cp_launch_plan(cp)
    rows = lambda i: slice(i * c, (i + 1) * c)  # noqa: E731
    # forward
    run_o, run_l2, o, lse = {}, {}, np.full_like(o_ref, np.nan), np.full_like(lse_ref, np.nan)
    for _, i, j, mq, _ in plan:
        o_p, lse_p = _partial(q[rows(i)], k[rows(j)], v[rows(j)], i * c, j * c, i == j)
        l2_p = lse_p / np.log(2.0)
        if mq & MERGE:
            mx = np.maximum(run_l2[i], l2_p)
            l2 = mx + np.log2(np.exp2(run_l2[i] - mx) + np.exp2(l2_p - mx))
            o_m = np.exp2(run_l2[i] - l2)[:, None] * run_o[i] + np.exp2(l2_p - l2)[:, None] * o_p
        else:
            l2, o_m = l2_p, o_p
        if mq & FINAL:
            o[rows(i)], lse[rows(i)] = o_m, l2 * np.log(2.0)
        else:
            run_o[i], run_l2[i] = o_m, l2
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)
    # backward: every pair from the merged LSE and delta = rowsum(dO * O)
    delta = (do * o).sum(axis=1)
    out = {n: np.full_like(q, np.nan) for n in ("dq", "dk", "dv")}
    run = {}
    for _, i, j, mq, mk in plan:
        qi, kj, vj, doi = q[rows(i)], k[rows(j)], v[rows(j)], do[rows(i)]
        sc = qi @ kj.T / np.sqrt(d)
        if i == j:
            sc = np.where(np.tril(np.ones((c, c), bool)), sc, -np.inf)
        p = np.exp(sc - lse[rows(i)][:, None])
        ds = p * (doi @ vj.T - delta[rows(i)][:, None])
        shares = (("dq", i, mq, ds @ kj / np.sqrt(d)), ("dk", j, mk, ds.T @ qi / np.sqrt(d)),
                  ("dv", j, mk, p.T @ doi))
        for name, chunk, mode, val in shares:
            acc = run[(name, chunk)] + val if mode & MERGE else val
            if mode & FINAL:
                out[name][rows(chunk)] = acc
            else:
                run[(name, chunk)] = acc
    for name, ref in (("dq", dq_ref), ("dk", dk_ref), ("dv", dv_ref)):
        np.testing.assert_allclose(out[name], ref, rtol=1e-12, atol=1e-12, err_msg=name)
