"""Helpers for GPU parity tests: drive the C ABI on a workload and compare each
stage with the CPU oracle. Imported only by tests (GPU tests and the benchmark's
parity sampling)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as WL


def config_for(mp, wl: WL.Workload, threshold: int = 2, match_mode: int = 0, centering: bool = True,
               center_query: bool = False):
    return mp.make_config(layers=wl.layers, batch=wl.batch, kv_heads=wl.kv_heads, q_heads=wl.q_heads,
                          head_dim=wl.head_dim, K=wl.K, L=wl.L, n_sink=wl.n_sink, window=wl.window,
                          capacity=wl.capacity, dtype=wl.dtype, w_per_layer=wl.w_per_layer,
                          threshold=threshold, match_mode=match_mode, centering=centering,
                          center_query=center_query)


class DeviceRun:
    """Buffers and calls for one workload on one device."""

    def __init__(self, mp, wl: WL.Workload, tensors: dict, device, threshold: int = 2, match_mode: int = 0,
                 centering: bool = True, center_query: bool = False):
        self.mp, self.wl, self.dev = mp, wl, torch.device(device)
        self.threshold = threshold
        self.cfg = config_for(mp, wl, threshold, match_mode, centering, center_query)
        self.tl = mp.mp_tables_layout_get(self.cfg)
        self.dl = mp.mp_decode_layout_get(self.cfg)
        self.tables = torch.empty(self.tl.total_bytes, dtype=torch.uint8, device=self.dev)
        self.scratch = torch.empty(self.dl.total_bytes, dtype=torch.uint8, device=self.dev)
        self.keys = tensors["keys"].to(self.dev)
        self.values = tensors["values"].to(self.dev)
        self.W = tensors["W"].to(self.dev).contiguous()
        self.queries = tensors["queries"].to(self.dev)
        self.out = torch.empty(wl.layers, wl.batch, wl.q_heads, wl.head_dim, dtype=torch.float32,
                               device=self.dev)

    def build(self):
        self.mp.mp_build_tables(self.cfg, self.keys, self.wl.n_prefill, self.W, self.tables)

    def append(self, pos: int):
        self.mp.mp_append(self.cfg, self.tables, self.keys, pos)

    def decode(self, step: int, n: int):
        q = self.queries[step].contiguous()
        self.mp.mp_decode_attention(self.cfg, self.tables, self.keys, self.values, n, q, self.out,
                                    self.scratch)
        return self.out

    def step(self, step: int, n: int):
        """Append token n - 1 and decode over n tokens in one call (mp_decode_step)."""
        q = self.queries[step].contiguous()
        self.mp.mp_decode_step(self.cfg, self.tables, self.keys, self.values, n - 1, q, self.out, self.scratch)
        return self.out

    def status(self) -> int:
        return self.mp.mp_get_status(self.tables)

    # ---- views (copied to host as numpy int64) ----
    def _view(self, buf, off, count, dtype):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return buf[off: off + nbytes].view(dtype)

    def codes(self) -> np.ndarray:
        wl = self.wl
        U = wl.layers * wl.batch * wl.kv_heads
        v = self._view(self.tables, self.tl.codes, U * wl.L * wl.capacity, torch.int16)
        return v.cpu().numpy().astype(np.int64).reshape(U, wl.L, wl.capacity) & 0xFFFF

    def unit_codes(self, u: int, n: int) -> np.ndarray:
        """Codes of tokens [0, n) of unit u, [n, L]."""
        wl = self.wl
        rows = []
        for t in range(wl.L):
            off = self.tl.codes + ((u * wl.L + t) * wl.capacity) * 2
            rows.append(self.tables[off: off + n * 2].view(torch.int16))
        v = torch.stack(rows).cpu().numpy().astype(np.int64) & 0xFFFF
        return v.T.copy()

    def unit_csr(self, u: int, tables: int):
        """Bucketed tables of unit u for the first `tables` tables: offsets
        [tables, NS, NB+1] and ids [tables, capacity] (16-bit, segment-local)."""
        wl = self.wl
        nb, ns = self.tl.n_buckets, -(-wl.capacity // 32768)
        o0 = self.tl.csr_offsets + u * wl.L * ns * (nb + 1) * 2
        i0 = self.tl.csr_ids + u * wl.L * wl.capacity * 2
        off = self.tables[o0: o0 + tables * ns * (nb + 1) * 2].view(torch.int16)
        ids = self.tables[i0: i0 + tables * wl.capacity * 2].view(torch.int16)
        return ((off.cpu().numpy().astype(np.int64) & 0xFFFF).reshape(tables, nb + 1, ns).transpose(0, 2, 1),
                (ids.cpu().numpy().astype(np.int64) & 0xFFFF).reshape(tables, wl.capacity))

    def unit_planes(self, u: int, tables: int) -> np.ndarray:
        """Bit-planes of unit u for the first `tables` tables, [tables, K, CW] as int64."""
        wl, cw = self.wl, self.tl.cap_words
        o = self.tl.planes + u * wl.L * wl.K * cw * 4
        v = self.tables[o: o + tables * wl.K * cw * 4].view(torch.int32)
        return (v.cpu().numpy().astype(np.int64) & 0xFFFFFFFF).reshape(tables, wl.K, cw)

    def center(self) -> np.ndarray:
        wl = self.wl
        U = wl.layers * wl.batch * wl.kv_heads
        return self._view(self.tables, self.tl.center, U * wl.head_dim, torch.float32).cpu().numpy().reshape(
            U, wl.head_dim)

    def decode_state(self):
        wl = self.wl
        Q = wl.layers * wl.batch * wl.q_heads
        qc = self._view(self.scratch, self.dl.q_codes, Q * wl.L, torch.int16).cpu().numpy().astype(np.int64)
        ln = self._view(self.scratch, self.dl.list_len, Q, torch.int32).cpu().numpy().astype(np.int64)
        ns = self._view(self.scratch, self.dl.sample_count, Q, torch.int32).cpu().numpy().astype(np.int64)
        return qc.reshape(Q, wl.L) & 0xFFFF, ln, ns

    def list_of(self, qh: int, length: int) -> np.ndarray:
        off = self.dl.lists + qh * self.wl.capacity * 4
        v = self.scratch[off: off + length * 4].view(torch.int32).cpu().numpy().astype(np.int64)
        return v & 0xFFFFFFFF


# ----------------------------------------------------------------------------------
# comparisons
# ----------------------------------------------------------------------------------

def tie_codes(ties: np.ndarray, K: int, L: int) -> np.ndarray:
    """Pack a near-tie mask [n, K*L] into per-table K-bit masks [n, L]."""
    out = np.zeros((ties.shape[0], L), dtype=np.int64)
    for t in range(L):
        for b in range(K):
            out[:, t] |= ties[:, t * K + b].astype(np.int64) << b
    return out


def compare_codes(gpu: np.ndarray, ref: np.ndarray, tiec: np.ndarray) -> dict:
    """gpu, ref, tiec: [n, L]. Every differing bit must be a near-tie bit."""
    diff = gpu ^ ref
    bad = (diff & ~tiec) != 0
    return {"bad": int(bad.sum()), "differ": int((diff != 0).sum()), "tie_bits": int(
        sum(bin(int(x)).count("1") for x in tiec[tiec != 0])) if tiec.any() else 0}


def unit_index(wl, layer, b, h):
    return (layer * wl.batch + b) * wl.kv_heads + h


def q_index(wl, layer, b, j):
    return (layer * wl.batch + b) * wl.q_heads + j


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def check_csr(off: np.ndarray, ids: np.ndarray, codes: np.ndarray, lo: int, hi: int, nb: int,
              seg: int = 32768) -> None:
    """Bucketed segments of one table against the (GPU) codes they were built from:
    in segment s (tokens [lo + s*seg, ...)), bucket b holds exactly the tokens with
    code b, stored as offsets from the segment's first token. The order inside a
    bucket is not unique (the build places tokens with shared-memory atomics), so
    the check is: the ids of a segment are a permutation of its tokens and the codes
    they point at, read in id order, are the bucket numbers the offsets give."""
    for si, a in enumerate(range(lo, hi, seg)):
        b = min(hi, a + seg)
        c = codes[a:b]
        o = off[si]
        counts = np.bincount(c, minlength=nb)
        assert o[0] == 0 and o[nb] == b - a
        np.testing.assert_array_equal(np.diff(o), counts)
        got = ids[si * seg: si * seg + (b - a)]
        np.testing.assert_array_equal(np.sort(got), np.arange(b - a))
        np.testing.assert_array_equal(c[got], np.repeat(np.arange(nb), counts))


# ----------------------------------------------------------------------------------
# end-to-end check of one workload
# ----------------------------------------------------------------------------------

def host_unit(tensors, wl, layer, b, h, n):
    k = tensors["keys"][layer, b, h, :n].double().cpu().numpy()
    v = tensors["values"][layer, b, h, :n].double().cpu().numpy()
    return k, v


def check_planes(planes: np.ndarray, codes: np.ndarray, n: int, K: int) -> None:
    """Bit-planes [K, CW] of one table against codes [n] of tokens [0, n)."""
    for b in range(K):
        bits = (planes[b][:, None] >> np.arange(32)[None, :]) & 1
        np.testing.assert_array_equal(bits.reshape(-1)[:n], (codes[:n] >> b) & 1)


def check_workload(mp, wl: WL.Workload, tensors: dict, device="cuda:0", threshold: int = 2,
                   units=None, qheads=None, steps=None, check_csr_tables: int = 8, tol: float = 2e-3,
                   match_mode: int = 0, centering: bool = True, center_query: bool = False,
                   use_step: bool = False) -> dict:
    """Build, append and decode `wl` through the C ABI and compare every stage with the
    oracle on the chosen units / query heads / steps. With center_query the query is
    hashed as q - c and p is the collision probability of q - c with k - c (the oracle's
    other reading). With use_step (appending workloads) every step is one mp_decode_step
    call instead of mp_append + mp_decode_attention. Returns counters for reporting."""
    run = DeviceRun(mp, wl, tensors, device, threshold, match_mode, centering, center_query)
    run.build()
    torch.cuda.synchronize()
    # the W status bit is informational (the tensor-core paths then use W's three-term split)
    assert (run.status() & ~mp.MP_STATUS_W_NOT_BF16) == 0, hex(run.status())
    U = wl.layers * wl.batch * wl.kv_heads
    all_units = [(l, b, h) for l in range(wl.layers) for b in range(wl.batch) for h in range(wl.kv_heads)]
    units = all_units if units is None else units
    steps = list(range(wl.steps)) if steps is None else steps
    rep = {"code_bits_tie": 0, "codes_differ": 0, "q_codes_differ": 0, "heads": 0, "max_rel_l2": 0.0,
           "sampled": 0, "region": 0, "S_differ_oracle_codes": 0, "match_mode": int(run.tl.match_mode)}
    n_tot = wl.capacity
    oracle_tabs = {}
    centers = run.center()
    for (l, b, h) in units:
        u = unit_index(wl, l, b, h)
        k64 = tensors["keys"][l, b, h, :n_tot].double().cpu().numpy()
        W64 = tensors["W"][l if wl.w_per_layer else 0].double().cpu().numpy()
        tab = O.HeadTables(k64, W64, wl.K, wl.L, wl.n_sink, wl.n_prefill, n_total=n_tot, centering=centering)
        oracle_tabs[u] = tab
        tiec = tie_codes(tab.ties, wl.K, wl.L)
        n0 = wl.n_prefill
        cmp = compare_codes(run.unit_codes(u, n0), tab.codes[:n0], tiec[:n0])
        assert cmp["bad"] == 0, (u, cmp)
        rep["codes_differ"] += cmp["differ"]
        rep["code_bits_tie"] += cmp["tie_bits"]
        np.testing.assert_allclose(centers[u], tab.center, rtol=1e-5, atol=1e-5)
        lo = min(wl.n_sink, n0)
        nt = min(wl.L, check_csr_tables)
        gc = run.unit_codes(u, n0)
        if run.tl.match_mode == mp.MP_MATCH_CSR:
            off, ids = run.unit_csr(u, nt)
            for t in range(nt):
                check_csr(off[t], ids[t], gc[:, t], lo, n0, run.tl.n_buckets)
        else:
            pl = run.unit_planes(u, nt)
            for t in range(nt):
                check_planes(pl[t], gc[:, t], n0, wl.K)
    last = max(steps) if steps else -1
    for step in range(last + 1):
        n = wl.seq_len(step)
        if wl.append and use_step:
            out_t = run.step(step, n)
        else:
            if wl.append:
                run.append(n - 1)
            out_t = run.decode(step, n)
        if step not in steps:
            continue
        out = out_t.cpu().numpy()
        torch.cuda.synchronize()
        st = run.status()
        assert (st & ~mp.MP_STATUS_W_NOT_BF16) == 0, hex(st)
        qc, ln, ns = run.decode_state()
        for (l, b, h) in units:
            u = unit_index(wl, l, b, h)
            tab = oracle_tabs[u]
            kc = run.unit_codes(u, n)
            if wl.append and run.tl.match_mode == mp.MP_MATCH_SCAN:
                pl = run.unit_planes(u, min(wl.L, check_csr_tables))
                for t in range(pl.shape[0]):
                    check_planes(pl[t], kc[:, t], n, wl.K)
            if wl.append:
                tiec = tie_codes(tab.ties[n - 1: n], wl.K, wl.L)
                cmp = compare_codes(kc[n - 1: n], tab.codes[n - 1: n], tiec)
                assert cmp["bad"] == 0, ("appended", u, n - 1, cmp)
                rep["codes_differ"] += cmp["differ"]
            k64, v64 = host_unit(tensors, wl, l, b, h, n)
            for g in range(wl.group):
                j = h * wl.group + g
                if qheads is not None and j not in qheads:
                    continue
                qi = q_index(wl, l, b, j)
                q64 = tensors["queries"][step, l, b, j].double().cpu().numpy()
                qh64 = q64 - tab.center if center_query else q64   # the hashed query
                W64 = tab.W
                qref = O.simhash_codes(qh64[None, :], W64, wl.K, wl.L)[0]
                qtie = tie_codes(O.near_ties(qh64[None, :], W64), wl.K, wl.L)[0]
                cq = compare_codes(qc[qi][None, :], qref[None, :], qtie[None, :])
                assert cq["bad"] == 0, ("query", qi, cq)
                rep["q_codes_differ"] += cq["differ"]
                # sampled set from the GPU's own codes: an integer function, exact
                counts = O.match_counts(kc, qc[qi])
                S_ref = O.sampled_set(counts, n, wl.n_sink, wl.window, threshold)
                lst = run.list_of(qi, int(ln[qi]))
                nsq = int(ns[qi])
                np.testing.assert_array_equal(lst[:nsq], S_ref)
                T_ref = O.exact_tokens(n, wl.n_sink, wl.window)
                assert np.all(lst[nsq:] & mp.EXACT_FLAG)
                np.testing.assert_array_equal(lst[nsq:] & ~mp.EXACT_FLAG, T_ref)
                # attention given S (oracle u, fp64) vs GPU output
                p = O.collision_probability(qh64, k64[S_ref] - tab.center[None, :])
                uS = O.inclusion_probability(p, wl.K, wl.L, threshold)
                o_ref = O.snis_attention(q64, k64, v64, S_ref, uS, T_ref)
                err = rel_l2(out[l, b, j], o_ref)
                assert err < tol, ("output", qi, err)
                rep["max_rel_l2"] = max(rep["max_rel_l2"], err)
                # the oracle end to end, with its own codes
                r = O.decode_head(q64, k64, v64, tab, n, wl.window, threshold, center_query=center_query)
                if not np.array_equal(r["S"], S_ref):
                    rep["S_differ_oracle_codes"] += 1
                    assert cq["differ"] > 0 or rep["codes_differ"] > 0, ("S differs without ties", qi)
                else:
                    assert rel_l2(out[l, b, j], r["out"]) < tol
                rep["heads"] += 1
                rep["sampled"] += nsq
                rep["region"] += max(0, n - wl.window - min(wl.n_sink, n))
    return rep
