"""Pins for the attention oracle: checks against things other than the oracle itself.

Each pin returns a list of failure messages (empty = pass), so the same pins can
be run against the real oracle (all must pass) and against planted-fault builds
of it (at least one must fail).  Inputs are drawn here, densely per request, and
then scattered into a shuffled page pool, so the library references never see
pages or block tables.
"""

from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

import oracle


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def dense_problem(seed, seq_lens, q_lens, *, Hq, Hkv, D, bs, shared_tokens=0, scale=None,
                  k_const=None, q_zero=False):
    """Draw per-request dense Q/K/V (bf16), then page them into a shuffled pool.

    The first ``shared_tokens`` tokens are identical across requests and are stored
    once, in blocks that every request's table points at (partial shared blocks are
    not shared physically).  Returns (paged dict for the oracle, dense dict).
    """
    g = torch.Generator().manual_seed(seed)
    n = len(seq_lens)
    shared_full = shared_tokens // bs
    shared_k = _bf16(torch.randn((shared_tokens, Hkv, D), generator=g))
    shared_v = _bf16(torch.randn((shared_tokens, Hkv, D), generator=g))
    dense_k, dense_v, dense_q = [], [], []
    for r in range(n):
        s = seq_lens[r]
        kk = _bf16(torch.randn((s, Hkv, D), generator=g))
        vv = _bf16(torch.randn((s, Hkv, D), generator=g))
        m = min(s, shared_tokens)
        kk[:m] = shared_k[:m]
        vv[:m] = shared_v[:m]
        if k_const is not None:
            kk[:] = k_const
        dense_k.append(kk)
        dense_v.append(vv)
        qq = _bf16(torch.randn((q_lens[r], Hq, D), generator=g))
        if q_zero:
            qq.zero_()
        dense_q.append(qq)
    used = [-(-s // bs) for s in seq_lens]
    private = [u - min(u, shared_full) for u in used]
    num_blocks = shared_full + sum(private) + 3
    perm = torch.randperm(num_blocks, generator=g).numpy()
    k_cache = torch.full((num_blocks, bs, Hkv, D), float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full((num_blocks, bs, Hkv, D), float("nan"), dtype=torch.bfloat16)
    width = max(used) + 1
    table = np.full((n, width), perm[-1], dtype=np.int32)
    cursor = shared_full
    for r in range(n):
        for b in range(used[r]):
            if b < shared_full:
                blk = perm[b]
            else:
                blk = perm[cursor]
                cursor += 1
            table[r, b] = blk
            lo, hi = b * bs, min((b + 1) * bs, seq_lens[r])
            k_cache[blk, : hi - lo] = dense_k[r][lo:hi]
            v_cache[blk, : hi - lo] = dense_v[r][lo:hi]
    q = torch.cat(dense_q, 0) if dense_q else torch.zeros((0, Hq, D), dtype=torch.bfloat16)
    cu = np.zeros(n + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    paged = dict(q=q, k_cache=k_cache, v_cache=v_cache, block_table=table, cu_seqlens_q=cu,
                 seq_lens=np.asarray(seq_lens, np.int32),
                 scale=scale if scale is not None else 1.0 / math.sqrt(D))
    dense = dict(q=dense_q, k=dense_k, v=dense_v, Hq=Hq, Hkv=Hkv, D=D)
    return paged, dense


def library_reference(paged, dense, lo_of=None, hi_of=None):
    """Dense attention per request with numpy matmul and scipy logsumexp/softmax.

    Key range of query i of request r (absolute position p): [lo_of(r, p), hi_of(r, p))
    with defaults [0, p + 1) (standard causal attention).
    """
    Hq, Hkv, D = dense["Hq"], dense["Hkv"], dense["D"]
    group = Hq // Hkv
    scale = paged["scale"]
    outs, lses = [], []
    for r, (qq, kk, vv) in enumerate(zip(dense["q"], dense["k"], dense["v"])):
        ql, s = qq.shape[0], kk.shape[0]
        qf = qq.double().numpy()            # [ql, Hq, D]
        kf = kk.double().numpy()            # [s, Hkv, D]
        vf = vv.double().numpy()
        pos = s - ql + np.arange(ql)        # absolute positions of the queries
        j = np.arange(s)
        lo = np.array([0 if lo_of is None else lo_of(r, p) for p in pos])
        hi = np.array([p + 1 if hi_of is None else hi_of(r, p) for p in pos])
        mask = (j[None, :] >= lo[:, None]) & (j[None, :] < hi[:, None])   # [ql, s]
        o = np.zeros((ql, Hq, D))
        l = np.full((ql, Hq), -np.inf)
        for h in range(Hq):
            gi = h // group
            S = scale * (qf[:, h, :] @ kf[:, gi, :].T)                     # [ql, s]
            S = np.where(mask, S, -np.inf)
            rows = mask.any(axis=1)
            l[rows, h] = scipy.special.logsumexp(S[rows], axis=1)
            P = np.zeros_like(S)
            P[rows] = scipy.special.softmax(S[rows], axis=1)
            o[:, h, :] = P @ vf[:, gi, :]
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def _run(paged, mutant, **kw):
    return oracle.attention(paged["q"], paged["k_cache"], paged["v_cache"], paged["block_table"],
                            paged["cu_seqlens_q"], paged["seq_lens"], paged["scale"],
                            mutant=mutant, n_threads=2, **kw)


def _close(a, b, tol, what):
    a = np.asarray(a)
    b = np.asarray(b)
    if a.shape != b.shape:
        return [f"{what}: shape {a.shape} vs {b.shape}"]
    fin = np.isfinite(b)
    if not np.array_equal(np.isfinite(a), fin):
        return [f"{what}: finiteness differs"]
    if not np.array_equal(a[~fin], b[~fin], equal_nan=True):
        return [f"{what}: non-finite values differ"]
    err = np.max(np.abs(a[fin] - b[fin]), initial=0.0)
    return [] if err <= tol else [f"{what}: max err {err:.3e} > {tol:.1e}"]


# -- pins -------------------------------------------------------------------------

CASES = [
    # (seed, seq_lens, q_lens, Hq, Hkv, D, bs, shared)
    (1, [5, 9, 17], [1, 3, 17], 4, 2, 8, 4, 4),
    (2, [33, 40], [8, 1], 8, 2, 16, 16, 16),
    (3, [20, 20, 20, 21], [1, 2, 5, 1], 6, 3, 32, 1, 12),
    (4, [64], [64], 4, 1, 16, 32, 0),
]


def pin_dense_library(mutant=0):
    """Standard attention equals dense numpy/scipy attention (bottom-right causal)."""
    fails = []
    for seed, sl, ql, Hq, Hkv, D, bs, sh in CASES:
        paged, dense = dense_problem(seed, sl, ql, Hq=Hq, Hkv=Hkv, D=D, bs=bs, shared_tokens=sh)
        ref_o, ref_l = library_reference(paged, dense)
        o, l = _run(paged, mutant)
        fails += _close(o, ref_o, 1e-10, f"case{seed} out")
        fails += _close(l, ref_l, 1e-10, f"case{seed} lse")
    return fails


def pin_partials_library(mutant=0):
    """Prefix phase (keys [0, c), non-causal) and suffix phase (keys [c, p]) equal the
    dense library attention restricted to those key ranges."""
    fails = []
    for seed, sl, ql, Hq, Hkv, D, bs, sh in CASES:
        paged, dense = dense_problem(seed, sl, ql, Hq=Hq, Hkv=Hkv, D=D, bs=bs, shared_tokens=sh)
        c = min(s - q for s, q in zip(sl, ql))
        ref_o, ref_l = library_reference(paged, dense, hi_of=lambda r, p: c)
        o, l = _run(paged, mutant, mode=oracle.PREFIX, cpl=c)
        fails += _close(o, ref_o, 1e-10, f"case{seed} prefix out")
        fails += _close(l, ref_l, 1e-10, f"case{seed} prefix lse")
        ref_o, ref_l = library_reference(paged, dense, lo_of=lambda r, p: c)
        o, l = _run(paged, mutant, mode=oracle.SUFFIX, cpl=c)
        fails += _close(o, ref_o, 1e-10, f"case{seed} suffix out")
        fails += _close(l, ref_l, 1e-10, f"case{seed} suffix lse")
    return fails


def pin_closed_forms(mutant=0):
    """One key: out = v, lse = scale q.k.  Zero query: out = mean(v), lse = ln n.
    Equal keys: out = mean(v), lse = scale q.k + ln n."""
    fails = []
    # one key
    paged, dense = dense_problem(11, [1], [1], Hq=2, Hkv=1, D=16, bs=16)
    o, l = _run(paged, mutant)
    v0 = dense["v"][0][0, 0].double().numpy()
    k0 = dense["k"][0][0, 0].double().numpy()
    for h in range(2):
        qh = dense["q"][0][0, h].double().numpy()
        fails += _close(o[0, h], v0, 0.0, "one-key out")
        fails += _close(l[0, h], paged["scale"] * float(np.dot(qh, k0)), 1e-14, "one-key lse")
    # zero query: uniform weights over the p + 1 visible keys
    sl, ql = [7, 12], [3, 2]
    paged, dense = dense_problem(12, sl, ql, Hq=4, Hkv=2, D=8, bs=4, q_zero=True)
    o, l = _run(paged, mutant)
    t = 0
    for r in range(2):
        vv = dense["v"][r].double().numpy()
        for i in range(ql[r]):
            p = sl[r] - ql[r] + i
            for h in range(4):
                fails += _close(o[t, h], vv[: p + 1, h // 2].mean(0), 1e-12, "zero-q out")
                fails += _close(l[t, h], math.log(p + 1), 1e-12, "zero-q lse")
            t += 1
    # all keys equal: same score everywhere
    kconst = _bf16(torch.linspace(-1, 1, 8)).expand(2, 8).clone()
    paged, dense = dense_problem(13, [9], [2], Hq=4, Hkv=2, D=8, bs=4, k_const=kconst)
    o, l = _run(paged, mutant)
    vv = dense["v"][0].double().numpy()
    for i in range(2):
        p = 9 - 2 + i
        for h in range(4):
            qh = dense["q"][0][i, h].double().numpy()
            s = paged["scale"] * float(np.dot(qh, kconst[h // 2].double().numpy()))
            fails += _close(o[i, h], vv[: p + 1, h // 2].mean(0), 1e-12, "equal-k out")
            fails += _close(l[i, h], s + math.log(p + 1), 1e-12, "equal-k lse")
    return fails


def pin_merge_identity(mutant=0):
    """merge(prefix phase, suffix phase) equals the standard path for every split point
    c <= min computed tokens; a -inf partner leaves the other partial unchanged."""
    fails = []
    sl, ql = [20, 26, 31], [2, 5, 1]
    paged, _ = dense_problem(21, sl, ql, Hq=4, Hkv=2, D=16, bs=4, shared_tokens=16)
    full_o, full_l = _run(paged, mutant)
    for c in range(0, min(s - q for s, q in zip(sl, ql)) + 1, 3):
        po, pl = _run(paged, mutant, mode=oracle.PREFIX, cpl=c)
        so, sl_ = _run(paged, mutant, mode=oracle.SUFFIX, cpl=c)
        mo, ml = oracle.merge_states(po, pl, so, sl_, mutant=mutant)
        fails += _close(mo, full_o, 1e-12, f"merge c={c} out")
        fails += _close(ml, full_l, 1e-12, f"merge c={c} lse")
    # -inf partner
    rng = np.random.default_rng(5)
    o1 = rng.standard_normal((6, 8))
    l1 = rng.standard_normal(6)
    o2 = np.zeros((6, 8))
    l2 = np.full(6, -np.inf)
    mo, ml = oracle.merge_states(o1, l1, o2, l2, mutant=mutant)
    fails += _close(mo, o1, 1e-15, "merge -inf out")
    fails += _close(ml, l1, 1e-15, "merge -inf lse")
    # both empty
    mo, ml = oracle.merge_states(o2, l2, o2, l2, mutant=mutant)
    fails += _close(mo, o2, 0.0, "merge empty out")
    fails += _close(ml, l2, 0.0, "merge empty lse")
    return fails


def pin_page_invariance(mutant=0):
    """Same logical KV, laid out with block sizes 1, 16 and 32 and shuffled pools:
    bit-identical results (the oracle sums in logical key order)."""
    fails = []
    sl, ql = [45, 50, 37], [3, 1, 6]
    ref = None
    for bs in (1, 16, 32):
        paged, _ = dense_problem(31, sl, ql, Hq=4, Hkv=2, D=16, bs=bs, shared_tokens=32)
        got = _run(paged, mutant)
        if ref is None:
            ref = got
        else:
            fails += _close(got[0], ref[0], 0.0, f"bs={bs} out")
            fails += _close(got[1], ref[1], 0.0, f"bs={bs} lse")
    return fails


def library_reference_sinks(paged, dense, sinks):
    """Dense attention with one more key per head: the sink logit s_h as an extra score
    column whose value row is zero, through scipy logsumexp / softmax."""
    Hq, Hkv, D = dense["Hq"], dense["Hkv"], dense["D"]
    group = Hq // Hkv
    scale = paged["scale"]
    outs, lses = [], []
    for qq, kk, vv in zip(dense["q"], dense["k"], dense["v"]):
        ql, s = qq.shape[0], kk.shape[0]
        qf, kf, vf = qq.double().numpy(), kk.double().numpy(), vv.double().numpy()
        pos = s - ql + np.arange(ql)
        mask = np.arange(s)[None, :] <= pos[:, None]                      # [ql, s]
        o = np.zeros((ql, Hq, D))
        l = np.zeros((ql, Hq))
        for h in range(Hq):
            gi = h // group
            S = np.where(mask, scale * (qf[:, h, :] @ kf[:, gi, :].T), -np.inf)
            S = np.concatenate([S, np.full((ql, 1), sinks[h])], axis=1)   # the sink column
            Vx = np.concatenate([vf[:, gi, :], np.zeros((1, D))], axis=0)  # its zero value
            l[:, h] = scipy.special.logsumexp(S, axis=1)
            o[:, h, :] = scipy.special.softmax(S, axis=1) @ Vx
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs, 0), np.concatenate(lses, 0)


def pin_sinks(mutant=0):
    """Attention sinks: equal to dense library attention with the sink as one more
    score column of zero value; -inf sinks give the standard path bit for bit; one key
    and one sink in closed form; the merge of the standard path with an (O = 0,
    lse = s_h) partial."""
    fails = []
    rng = np.random.default_rng(41)
    for seed, sl, ql, Hq, Hkv, D, bs, sh in CASES:
        paged, dense = dense_problem(seed, sl, ql, Hq=Hq, Hkv=Hkv, D=D, bs=bs, shared_tokens=sh)
        sinks = rng.standard_normal(Hq) * 3.0
        sinks[0] = -np.inf
        ref_o, ref_l = library_reference_sinks(paged, dense, sinks)
        o, l = _run(paged, mutant, sinks=sinks)
        fails += _close(o, ref_o, 1e-10, f"case{seed} sinks out")
        fails += _close(l, ref_l, 1e-10, f"case{seed} sinks lse")
        # -inf everywhere: the standard path exactly
        so, sl_ = _run(paged, mutant, sinks=np.full(Hq, -np.inf))
        po, pl = _run(paged, mutant)
        fails += _close(so, po, 0.0, f"case{seed} -inf sinks out")
        fails += _close(sl_, pl, 0.0, f"case{seed} -inf sinks lse")
        # the sink as one more partial of the LSE merge
        t = l.shape[0]
        mo, ml = oracle.merge_states(po, pl, np.zeros_like(po),
                                     np.broadcast_to(sinks, pl.shape).copy(), mutant=mutant)
        fails += _close(mo, o, 1e-12, f"case{seed} sinks merge out")
        fails += _close(ml, l, 1e-12, f"case{seed} sinks merge lse")
    # one key x and one sink s: out = v e^x / (e^x + e^s), lse = ln(e^x + e^s)
    paged, dense = dense_problem(42, [1], [1], Hq=2, Hkv=1, D=16, bs=16)
    sinks = np.array([0.75, -2.5])
    o, l = _run(paged, mutant, sinks=sinks)
    v0 = dense["v"][0][0, 0].double().numpy()
    k0 = dense["k"][0][0, 0].double().numpy()
    for h in range(2):
        x = paged["scale"] * float(np.dot(dense["q"][0][0, h].double().numpy(), k0))
        w = 1.0 / (1.0 + math.exp(sinks[h] - x))
        fails += _close(o[0, h], v0 * w, 1e-14, "one key + sink out")
        fails += _close(l[0, h], x + math.log1p(math.exp(sinks[h] - x)), 1e-14,
                        "one key + sink lse")
    return fails


def to_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """x / scale as E4M3 bytes (torch's float8_e4m3fn rounding: input drawing only)."""
    return (x.float() / scale).to(torch.float8_e4m3fn).view(torch.uint8)


def e4m3_library_values() -> np.ndarray:
    """The 256 codes decoded by torch's float8_e4m3fn (a library routine)."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_fp8kv(mutant=0):
    """FP8 (E4M3) KV cache: every code decodes as torch's float8_e4m3fn does; over a
    cache whose scaled values are exact in bf16 (power-of-two scales) the FP8 oracle
    equals the bf16 oracle on those values bit for bit; with other scales it equals
    dense library attention over the decoded, scaled values."""
    fails = []
    got = oracle.e4m3_values(mutant=mutant)
    fails += _close(got, e4m3_library_values(), 0.0, "e4m3 code table")
    for seed, sl, ql, Hq, Hkv, D, bs, sh in CASES:
        paged, dense = dense_problem(seed, sl, ql, Hq=Hq, Hkv=Hkv, D=D, bs=bs, shared_tokens=sh)
        for ks, vs, exact in ((2.0 ** -4, 2.0 ** -3, True), (0.0173, 0.0291, False)):
            kb = to_e4m3(paged["k_cache"], ks)
            vb = to_e4m3(paged["v_cache"], vs)
            o, l = oracle.attention_fp8kv(paged["q"], kb, vb, paged["block_table"],
                                          paged["cu_seqlens_q"], paged["seq_lens"],
                                          paged["scale"], ks, vs, mutant=mutant, n_threads=2)
            kd = kb.view(torch.float8_e4m3fn).double() * ks
            vd = vb.view(torch.float8_e4m3fn).double() * vs
            if exact:
                ref = dict(paged, k_cache=kd.to(torch.bfloat16), v_cache=vd.to(torch.bfloat16))
                assert torch.equal(ref["k_cache"].double().nan_to_num(7.0), kd.nan_to_num(7.0))
                ro, rl = _run(ref, mutant)
                fails += _close(o, ro, 0.0, f"case{seed} fp8 vs bf16 out")
                fails += _close(l, rl, 0.0, f"case{seed} fp8 vs bf16 lse")
            else:
                # the dense requests' values, through the same quantisation
                dk = [(to_e4m3(k, ks).view(torch.float8_e4m3fn).double() * ks) for k in dense["k"]]
                dv = [(to_e4m3(v, vs).view(torch.float8_e4m3fn).double() * vs) for v in dense["v"]]
                ro, rl = library_reference(paged, dict(dense, k=dk, v=dv))
                fails += _close(o, ro, 1e-10, f"case{seed} fp8 library out")
                fails += _close(l, rl, 1e-10, f"case{seed} fp8 library lse")
    return fails


ALL_PINS = [pin_dense_library, pin_partials_library, pin_closed_forms, pin_merge_identity,
            pin_page_invariance, pin_sinks, pin_fp8kv]
