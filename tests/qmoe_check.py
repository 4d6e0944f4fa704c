"""Comparison helpers shared by the GPU parity tests (no method arithmetic).

Tolerance for layer outputs (fp16/bf16 out, fp32 accumulation):
    |gpu - ref| <= 1e-2 * (1 + |ref|) elementwise.
Routing: expert ids must equal the oracle's exactly, except for tokens whose
oracle k-th and (k+1)-th probabilities differ by less than 1e-4 ("near
ties"); for those the GPU's choice must still be a valid top-k within 1e-4,
and the output is compared with the oracle re-run on the GPU's routing.
"""
import numpy as np
import torch

TOL = 1e-2
NEAR_TIE = 1e-4
# Stricter than the near-tie rule: fp32 logits differ from fp64 by ~1e-8 in
# probability, so any token whose k-th / (k+1)-th gap exceeds this must
# match the oracle exactly too.
STRICT_GAP = 2e-6


def to_f64(t):
    return t.detach().float().cpu().double().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float64)


def assert_close_layer(got, ref, what=""):
    got = to_f64(got)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bound = TOL * (1.0 + np.abs(ref))
    bad = err > bound
    assert not bad.any(), "%s: %d elements out of tolerance, worst err %.4g at ref %.4g (max |ref| %.3g)" % (
        what, int(bad.sum()), float(err.max()), float(ref.flat[int(np.argmax(err - bound))]), float(np.abs(ref).max()))
    return float((err / (1.0 + np.abs(ref))).max())


def near_tie_tokens(probs, k):
    """Tokens whose k-th and (k+1)-th oracle probabilities are within NEAR_TIE."""
    s = -np.sort(-probs, axis=1)
    if probs.shape[1] <= k:
        return np.zeros(probs.shape[0], dtype=bool)
    return (s[:, k - 1] - s[:, k]) < NEAR_TIE


def check_routing(gpu_ids, gpu_w, probs, ref_ids, k):
    """Ids bit-exact outside near ties; near-tie choices valid within NEAR_TIE
    (and exact unless the gap is below STRICT_GAP).  Returns the boolean mask
    of near-tie tokens (gap < NEAR_TIE), the count the layer reports."""
    gpu_ids = np.asarray(gpu_ids)
    near = near_tie_tokens(probs, k)
    s_all = -np.sort(-probs, axis=1)
    strict_ok = (s_all[:, k - 1] - s_all[:, k]) >= STRICT_GAP if probs.shape[1] > k else np.ones(len(probs), bool)
    for t in range(probs.shape[0]):
        if not near[t] or strict_ok[t]:
            assert list(gpu_ids[t]) == list(ref_ids[t]), "token %d: ids %s vs oracle %s" % (
                t, list(gpu_ids[t]), list(ref_ids[t]))
        else:
            s = -np.sort(-probs[t])
            pk, pk1 = s[k - 1], s[k]
            chosen = set(int(e) for e in gpu_ids[t])
            assert len(chosen) == k
            for e in range(probs.shape[1]):
                if e in chosen:
                    assert probs[t, e] >= pk1 - NEAR_TIE
                else:
                    assert probs[t, e] <= pk + NEAR_TIE
    gw = np.asarray(gpu_w, np.float64)
    pw = np.take_along_axis(probs, gpu_ids.astype(np.int64), axis=1)
    np.testing.assert_allclose(gw, pw, rtol=1e-5, atol=1e-7)
    return near


def run_layer_and_check(wl, L, path, accumulate=False, seed=0):
    """Run one qmoe_forward through the C ABI on `path` and compare it with
    the fp64 oracle (routing with the near-tie rule, output elementwise).
    Returns (output, topk weights, topk ids, worst relative error, near-tie count)."""
    import oracle
    from int4_block_quantized_gb300 import binding as B
    x = L["x"]
    out0 = None
    out = None
    if accumulate:
        out0 = torch.randn(x.shape, generator=torch.Generator(device=x.device).manual_seed(seed + 7),
                           device=x.device).to(x.dtype)
        out = out0.clone()
    ws = B.Workspace(x.shape[0], wl.H, wl.I, wl.E, wl.k, device=x.device)
    o, tw, ti = B.qmoe_forward(L, out=out, ws=ws, accumulate=accumulate, path=path, return_routing=True)
    torch.cuda.synchronize()
    assert ws.status() == (0, 0)
    ref, ref_ids, ref_w, probs = oracle.qmoe_forward(L)
    ids = ti.cpu().numpy()
    near = check_routing(ids, tw.cpu().numpy(), probs, ref_ids, wl.k)
    if near.any():
        ref2, _, _, _ = oracle.qmoe_forward(L, forced_ids=ids, forced_w=tw.cpu().double().numpy())
        ref[near] = ref2[near]
    if accumulate:
        ref = ref + out0.double().cpu().numpy()
    return o, tw, ti, assert_close_layer(o, ref, wl.name), int(near.sum())


# ---- the oracle over many tokens, spread over the host's cores.  Each
# token's output depends only on that token, so token chunks are independent
# oracle calls.  Workers start by spawn (the test process already holds a
# CUDA context) and memory-map the layer's tensors from a temporary folder.
_TENSORS = ("x", "router_w", "router_bias", "gate_w", "gate_s", "gate_zp", "up_w", "up_s", "up_zp",
            "down_w", "down_s", "down_zp")
_INTS = ("T", "H", "I", "E", "k", "block_size", "act_dtype", "scale_dtype")


def _oracle_chunk(args):
    import os as _os
    import numpy as _np
    import oracle as _oracle
    folder, lo, hi, ints, present = args
    L = dict(ints)
    for n in present:
        a = _np.load(_os.path.join(folder, n + ".npy"), mmap_mode="r")
        L[n] = a[lo:hi] if n == "x" else a
    L["T"] = hi - lo
    out, ids, w, probs = _oracle.qmoe_forward(L)
    return lo, out, ids, w, probs


def oracle_forward_parallel(L, nproc=None):
    """oracle.qmoe_forward(L) over all of L's tokens, one contiguous chunk per
    process (each oracle call copies the whole layer's weights once, so
    fewer, larger chunks are faster).  Returns (out, ids, w, probs) like
    oracle.qmoe_forward."""
    import multiprocessing as mp
    import os
    import shutil
    import tempfile
    folder = tempfile.mkdtemp(prefix="qmoe_oracle_")
    try:
        present = []
        for n in _TENSORS:
            t = L.get(n)
            if t is None:
                continue
            if isinstance(t, torch.Tensor):
                t = t.detach().cpu().contiguous()
                if t.dtype in (torch.float16, torch.bfloat16):
                    t = t.view(torch.int16)
                t = t.numpy()
            np.save(os.path.join(folder, n + ".npy"), np.ascontiguousarray(t))
            present.append(n)
        ints = {n: int(L[n]) for n in _INTS}
        T = ints["T"]
        ncpu = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
        nproc = max(1, min(T, nproc or ncpu))
        chunk = -(-T // nproc)
        jobs = [(folder, lo, min(T, lo + chunk), ints, present) for lo in range(0, T, chunk)]
        with mp.get_context("spawn").Pool(nproc) as pool:
            parts = pool.map(_oracle_chunk, jobs)
        parts.sort(key=lambda r: r[0])
        return (np.concatenate([p[1] for p in parts]), np.concatenate([p[2] for p in parts]),
                np.concatenate([p[3] for p in parts]), np.concatenate([p[4] for p in parts]))
    finally:
        shutil.rmtree(folder, ignore_errors=True)


def tile_columns(ids, E, tile=160):
    """Column of every assignment (token t, slot j) inside its expert's token
    tile, for routing ids [T, k]: assignments are grouped by expert in
    (token, slot) order, and an expert with n assignments is one tile when
    n <= tile, else ceil(n / 128) tiles of ceil(n / tiles) rows.  Returns
    [T, k] ints."""
    ids = np.asarray(ids)
    T, k = ids.shape
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    rank = np.zeros(flat.size, dtype=np.int64)
    seen = np.zeros(E, dtype=np.int64)
    for a, e in enumerate(flat):
        rank[a] = seen[e]
        seen[e] += 1
    # one tile when n <= tile, else ceil(n / 128) tiles of balanced size
    ntile = np.where(counts <= tile, (counts > 0).astype(np.int64), (counts + 127) // 128)
    rows = np.where(ntile > 0, (counts + np.maximum(ntile, 1) - 1) // np.maximum(ntile, 1), 1)
    return (rank % rows[flat]).reshape(T, k)


def tokens_covering_tile_columns(ids, E, n_extra, seed, tile=160):
    """Token indices whose assignments together sit at every tile column
    that occurs (greedy), plus n_extra more drawn at random."""
    cols = tile_columns(ids, E, tile)
    T = cols.shape[0]
    need = set(int(c) for c in np.unique(cols))
    chosen = []
    for t in np.argsort([-len(set(r)) for r in cols.tolist()], kind="stable"):
        new = set(int(c) for c in cols[t]) & need
        if new:
            chosen.append(int(t))
            need -= new
        if not need:
            break
    rest = np.setdiff1d(np.arange(T), chosen)
    rng = np.random.default_rng(seed)
    extra = rng.choice(rest, size=min(n_extra, rest.size), replace=False).tolist()
    picked = sorted(set(chosen) | set(int(t) for t in extra))
    covered = set(int(c) for c in np.unique(cols[picked]))
    assert covered == set(int(c) for c in np.unique(cols)), "tile columns not all covered"
    return picked
