"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins
catch every one of them: a dropped term, a wrong sign or index, a transposed
or swapped operand, a wrong digit or bit order, a wrong plane offset."""
import numpy as np
import pytest

import oracle
import oracle.ternary as T
import pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(T, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _orig(name):
    return getattr(T, name)


def m_pq2_msb_first(mp):
    def dec(base_g):
        b = base_g.astype(np.int64)
        f = [((b >> (6 - 2 * i)) & 3) for i in range(4)]
        return np.stack(f, -1).reshape(base_g.shape[:-1] + (128,)) - 1
    _patch(mp, "_decode_pq2", dec)


def m_pq2_twos_complement(mp):
    def dec(base_g):
        b = base_g.astype(np.int64)
        f = [((b >> (2 * i)) & 3) for i in range(4)]
        c = np.stack(f, -1).reshape(base_g.shape[:-1] + (128,))
        return np.where(c >= 2, c - 4, c)
    _patch(mp, "_decode_pq2", dec)


def m_pq2_no_offset(mp):
    orig = _orig("_decode_pq2")
    _patch(mp, "_decode_pq2", lambda b: orig(b) + 1)


def m_ptq1_big_endian(mp):
    def dec(base_g, high_g):
        b = base_g.astype(np.int64)
        h = high_g.astype(np.int64)
        lead = base_g.shape[:-1]
        lo = np.stack([(b // 3 ** (4 - i)) % 3 for i in range(5)], -1).reshape(lead + (120,))
        hi = np.stack([(h // 3 ** (3 - i)) % 3 for i in range(4)], -1).reshape(lead + (8,))
        return np.concatenate([lo, hi], -1) - 1
    _patch(mp, "_decode_ptq1", dec)


def m_ptq1_high_first(mp):
    orig = _orig("_decode_ptq1")
    def dec(base_g, high_g):
        v = orig(base_g, high_g)
        return np.concatenate([v[..., 120:], v[..., :120]], -1)
    _patch(mp, "_decode_ptq1", dec)


def m_forward_no_normalisation(mp):
    orig = _orig("hadamard_forward")
    _patch(mp, "hadamard_forward", lambda x, s: orig(x, s) * 32.0)


def m_forward_signs_after(mp):
    _patch(mp, "hadamard_forward", _orig("hadamard_inverse"))


def m_inverse_signs_before(mp):
    _patch(mp, "hadamard_inverse", _orig("hadamard_forward"))


def m_signs_not_global(mp):
    orig = _orig("hadamard_forward")
    def fw(x, s):
        s = np.asarray(s, dtype=np.float64).reshape(-1)
        return orig(x, np.tile(s[:1024], s.size // 1024) if s.size % 1024 == 0 else s)
    _patch(mp, "hadamard_forward", fw)


def m_sequency_order(mp):
    orig = _orig("hadamard_matrix")
    def H(size=1024):
        h = orig(size)
        order = np.argsort((np.abs(np.diff(h, axis=1)) > 0).sum(axis=1), kind="stable")
        return h[order]
    _patch(mp, "hadamard_matrix", H)


def m_scale_offset_in_high_plane(mp):
    orig = _orig("row_split_geometry")
    def geo(fmt, n, k):
        g = orig(fmt, n, k)
        return g._replace(scale_offset=g.base_bytes)
    _patch(mp, "row_split_geometry", geo)


def m_high_offset_unaligned(mp):
    orig = _orig("row_split_geometry")
    def geo(fmt, n, k):
        g = orig(fmt, n, k)
        d = g.high_offset - g.base_bytes
        return g._replace(high_offset=g.base_bytes, scale_offset=g.scale_offset - d,
                          payload_bytes=g.payload_bytes - d)
    _patch(mp, "row_split_geometry", geo)


def m_kpad_not_aligned(mp):
    orig = _orig("row_split_geometry")
    def geo(fmt, n, k):
        g = orig(fmt, n, k)
        return g._replace(k_pad=k)
    _patch(mp, "row_split_geometry", geo)


def m_scale_wrong_group(mp):
    orig = _orig("dequantize")
    def deq(fmt, payload, n, k, rows=None):
        w = orig(fmt, payload, n, k, rows)
        return np.roll(w.reshape(w.shape[0], -1, 128), 1, axis=1).reshape(w.shape) if k % 128 == 0 else w
    _patch(mp, "dequantize", deq)


def m_scale_dropped(mp):
    orig = _orig("dequantize")
    def deq(fmt, payload, n, k, rows=None):
        w = orig(fmt, payload, n, k, rows)
        return np.sign(w)
    _patch(mp, "dequantize", deq)


def m_transform_dropped(mp):
    def mm(fmt, payload, n, k, x, signs=None, rows=None):
        x = np.atleast_2d(np.asarray(x, dtype=np.float64))
        return x @ T.dequantize(fmt, payload, n, k, rows).T
    _patch(mp, "ternary_matmul", mm)


def m_rows_reversed(mp):
    orig = _orig("ternary_matmul")
    _patch(mp, "ternary_matmul", lambda *a, **kw: orig(*a, **kw)[:, ::-1])


def m_embed_forward(mp):
    def emb(fmt, payload, n, k, ids, signs):
        return T.hadamard_forward(T.dequantize(fmt, payload, n, k, ids), signs)
    _patch(mp, "embed_rows", emb)


def m_blocks_scale_after(mp):
    monkeypatch_slices = dict(T.BLOCK_PLANE_SLICES)
    monkeypatch_slices["PQ2_0_G128"] = ((0, 32), None, (32, 34))
    mp.setattr(T, "BLOCK_PLANE_SLICES", monkeypatch_slices)


def m_blocks_ptq1_high_first(mp):
    # PTQ1_0 block read as [high 2][base 24][scale 2] instead of [base 24][high 2][scale 2]
    monkeypatch_slices = dict(T.BLOCK_PLANE_SLICES)
    monkeypatch_slices["PTQ1_0_G128"] = ((2, 26), (0, 2), (26, 28))
    mp.setattr(T, "BLOCK_PLANE_SLICES", monkeypatch_slices)


def m_pack_pad_minus_one(mp):
    orig = _orig("pack_planes")
    def pk(fmt, values, scales):
        values = np.asarray(values)
        n, k = values.shape
        kp = -(-k // 128) * 128
        if kp == k:
            return orig(fmt, values, scales)
        full = np.full((n, kp), -1, np.int8)
        full[:, :k] = values
        p = orig(fmt, full, scales)
        return p
    _patch(mp, "pack_planes", pk)


def m_swiglu_sigmoid_gate(mp):
    def f(fmt, pg, pu, n, k, x, sg=None, su=None, rows=None):
        g = T.ternary_matmul(fmt, pg, n, k, x, sg, rows)
        u = T.ternary_matmul(fmt, pu, n, k, x, su, rows)
        return 1.0 / (1.0 + np.exp(-g)) * u
    _patch(mp, "gate_up_swiglu", f)


def m_swiglu_operands_swapped(mp):
    orig = _orig("gate_up_swiglu")
    def f(fmt, pg, pu, n, k, x, sg=None, su=None, rows=None):
        return orig(fmt, pu, pg, n, k, x, su, sg, rows)
    _patch(mp, "gate_up_swiglu", f)


def m_swiglu_one_sign_vector(mp):
    orig = _orig("gate_up_swiglu")
    def f(fmt, pg, pu, n, k, x, sg=None, su=None, rows=None):
        return orig(fmt, pg, pu, n, k, x, sg, sg, rows)
    _patch(mp, "gate_up_swiglu", f)


def m_ptq1_invalid_bytes_to_zero(mp):
    # bytes the packer never writes (>= 243 base, >= 81 high) read as all-zero values
    orig = _orig("_decode_ptq1")
    def dec(base_g, high_g):
        v = orig(base_g, high_g)
        lead = base_g.shape[:-1]
        bad_lo = np.repeat(base_g >= 243, 5, axis=-1).reshape(lead + (120,))
        bad_hi = np.repeat(high_g >= 81, 4, axis=-1).reshape(lead + (8,))
        return np.where(np.concatenate([bad_lo, bad_hi], -1), 0, v)
    _patch(mp, "_decode_ptq1", dec)


def m_ptq1_fifth_digit_dropped(mp):
    # t4 of every base byte read as 0 (value -1): a four-digit reading of five
    orig = _orig("_decode_ptq1")
    def dec(base_g, high_g):
        v = orig(base_g, high_g).copy()
        v[..., 4:120:5] = -1
        return v
    _patch(mp, "_decode_ptq1", dec)


def m_error_abs_dropped(mp):
    def f(got, ref):
        got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
        den = np.max(np.abs(ref)) if ref.size else 0.0
        num = np.max(got - ref) if ref.size else 0.0
        return float(num / den) if den > 0 else float(num)
    _patch(mp, "max_rel_error", f)


def m_error_normalised_by_got(mp):
    def f(got, ref):
        got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
        den = np.max(np.abs(got)) if got.size else 0.0
        num = np.max(np.abs(got - ref)) if ref.size else 0.0
        return float(num / den) if den > 0 else float(num)
    _patch(mp, "max_rel_error", f)


def m_error_mean_not_max(mp):
    def f(got, ref):
        got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
        den = np.mean(np.abs(ref)) if ref.size else 0.0
        num = np.mean(np.abs(got - ref)) if ref.size else 0.0
        return float(num / den) if den > 0 else float(num)
    _patch(mp, "max_rel_error", f)


def m_error_zero_reference_scores_zero(mp):
    orig = _orig("max_rel_error")
    def f(got, ref):
        ref_a = np.asarray(ref, np.float64)
        return 0.0 if not np.any(ref_a) else orig(got, ref)
    _patch(mp, "max_rel_error", f)


def m_significant_threshold_on_max(mp):
    def f(got, ref, floor=0.1):
        got, ref = np.asarray(got, np.float64).reshape(-1), np.asarray(ref, np.float64).reshape(-1)
        if ref.size == 0 or not np.any(ref):
            return 0.0
        sel = np.abs(ref) >= floor * np.max(np.abs(ref))
        return float(np.max(np.abs(got[sel] - ref[sel]) / np.abs(ref[sel])))
    _patch(mp, "significant_rel_error", f)


def m_significant_normalised_by_max(mp):
    def f(got, ref, floor=0.1):
        got, ref = np.asarray(got, np.float64).reshape(-1), np.asarray(ref, np.float64).reshape(-1)
        if ref.size == 0 or not np.any(ref):
            return 0.0
        sel = np.abs(ref) >= floor * np.sqrt(np.mean(ref * ref))
        return float(np.max(np.abs(got[sel] - ref[sel])) / np.max(np.abs(ref)))
    _patch(mp, "significant_rel_error", f)


def m_significant_no_threshold(mp):
    def f(got, ref, floor=0.1):
        got, ref = np.asarray(got, np.float64).reshape(-1), np.asarray(ref, np.float64).reshape(-1)
        sel = ref != 0
        return float(np.max(np.abs(got[sel] - ref[sel]) / np.abs(ref[sel]))) if np.any(sel) else 0.0
    _patch(mp, "significant_rel_error", f)


MUTATIONS = [v for k, v in sorted(globals().items()) if k.startswith("m_")]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda f: f.__name__)
def test_mutation_is_caught(mutation, monkeypatch):
    mutation(monkeypatch)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin()
        except Exception as exc:  # an assertion or a shape/value error both count
            caught.append((pin.__name__, type(exc).__name__))
            break
    assert caught, f"no pin catches {mutation.__name__}"
