"""Plant plausible mistakes in a copy of the CPU oracle and check that the pins
catch every one of them (no GPU).  A mutant is a text substitution in the
oracle's source, loaded as a fresh module; the real oracle is never touched.
"""
import os
import types

import pytest

from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attention.py")

# (name, exact text in the oracle, replacement, how many occurrences to replace)
MUTANTS = [
    ("scale dropped", "s = scale * (q_rows @ k.T)", "s = (q_rows @ k.T)", 1),
    ("K not transposed", "s = scale * (q_rows @ k.T)", "s = scale * (q_rows @ k)", 1),
    ("mask off by one", "k_pos[None, :] > q_pos[:, None]", "k_pos[None, :] >= q_pos[:, None]", 1),
    ("mask transposed", "k_pos[None, :] > q_pos[:, None]", "k_pos[None, :] < q_pos[:, None]", 1),
    ("no max subtraction", "np.exp(s - m[:, None]), 0.0).astype(dtype)", "np.exp(s), 0.0).astype(dtype)", 1),
    ("exp sign flipped", "np.exp(s - m[:, None]), 0.0).astype(dtype)",
     "np.exp(m[:, None] - s), 0.0).astype(dtype)", 1),
    ("no division by l", "acc_or_e_v / np.where(empty, 1.0, l)[:, None]", "acc_or_e_v", 1),
    ("LSE without m", "m + np.log(np.where(empty, 1.0, l))", "np.log(np.where(empty, 1.0, l))", 1),
    ("LSE in log2", "m + np.log(np.where(empty, 1.0, l))", "m + np.log2(np.where(empty, 1.0, l))", 1),
    ("empty row gets NaN", "np.where(empty[:, None], 0.0, acc_or_e_v", "np.where(empty[:, None], np.nan, acc_or_e_v", 1),
    ("query offset ignored", "causal, q_offset + idx, k_pos)", "causal, idx, k_pos)", 1),
    ("key offset ignored", "k_pos = k_offset + np.arange(k.shape[0], dtype=np.int64)",
     "k_pos = np.arange(k.shape[0], dtype=np.int64)", 1),
    ("split merge weight sign", "np.exp(lse_s - np.where(seen, top, 0.0)[None, :])",
     "np.exp(np.where(seen, top, 0.0)[None, :] - lse_s)", 1),
    ("split merge ignores LSE_s", "np.exp(lse_s - np.where(seen, top, 0.0)[None, :])",
     "np.exp(0.0 * lse_s)", 1),
    ("split LSE drops total", "top + np.log(np.where(seen, total, 1.0))", "top + 0.0 * total", 1),
    ("bwd: D from dP instead of O", "d_row = (do * o).sum(axis=1)", "d_row = (do * v[: do.shape[0]]).sum(axis=1)", 1),
    ("bwd: softmax Jacobian sign", "ds = p * (dp - d_row[:, None])", "ds = p * (dp + d_row[:, None])", 1),
    ("bwd: D dropped", "ds = p * (dp - d_row[:, None])", "ds = p * dp", 1),
    ("bwd: dV not transposed", "dv = p.T @ do", "dv = p @ do", 1),
    ("bwd: dK scale dropped", "dk = scale * (ds.T @ q)", "dk = (ds.T @ q)", 1),
    ("bwd: dQ uses V", "dq = scale * (ds @ k)", "dq = scale * (ds @ v)", 1),
    ("split key offsets ignored", "rows=rows, q_offset=q_offset, k_offset=a))",
     "rows=rows, q_offset=q_offset, k_offset=0))", 1),
    ("P uses V", "return e / e.sum(axis=1)[:, None]", "return e / e.sum(axis=0)[None, :]", 1),
    ("rescale with tile max", "r = np.where(seen, np.exp(m - m_new), 0.0)",
     "r = np.where(seen, np.exp(m_ij - m_new), 0.0)", 1),
    ("rescale dropped from l", "l = r * l + p_ij.sum(axis=1)", "l = l + p_ij.sum(axis=1)", 1),
    ("rescale dropped from O~", "acc = r[:, None] * acc + p_ij @ v[a:b]", "acc = acc + p_ij @ v[a:b]", 1),
    ("block exp against tile max", "np.exp(s_ij - m_new[:, None])", "np.exp(s_ij - m_ij[:, None])", 1),
    ("running max not kept", "        m = m_new\n        if trace is not None:\n            with",
     "        if trace is not None:\n            with", 1),
    ("normalised: l factor dropped", "((a_old * ell)[:, None] * out", "((a_old)[:, None] * out", 1),
    ("normalised: new-block weight dropped", "a_new[:, None] * (p_t @ v[a:b])", "(p_t @ v[a:b])", 1),
    ("normalised: l~ not rescaled", "l_new = a_old * ell + a_new * l_t", "l_new = a_old * ell + l_t", 1),
    ("brute force: wrong LSE", "lse[i] = m + math.log(denom)", "lse[i] = math.log(denom)", 1),
    ("brute force: scale dropped", "s[j] = scale * dot", "s[j] = dot", 1),
    ("brute force: causal off by one", "if not (causal and k_offset + j > q_offset + i)",
     "if not (causal and k_offset + j >= q_offset + i)", 1),
]


def _load_mutant(old, new, count):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= count, f"mutation site not found: {old!r}"
    mutated = src.replace(old, new, count)
    mod = types.ModuleType("oracle_mutant")
    exec(compile(mutated, "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, count):
    mod = _load_mutant(old, new, count)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 -- any failure of a pin counts
            caught.append(pin.__name__)
    assert caught, f"mutant '{name}' passed every pin"


# ---------------------------------------------------------------- the FP8 oracle
from tests.oracle_pins_fp8 import FP8_PINS  # noqa: E402

FP8_SRC = os.path.join(os.path.dirname(SRC), "fp8.py")

FP8_MUTANTS = [
    ("e4m3 bias 8", "(1.0 + m / 8.0) * 2.0 ** (e - 7)", "(1.0 + m / 8.0) * 2.0 ** (e - 8)", 1),
    ("e4m3 keeps the NaN code", "if e == 15 and m == 7:", "if e == 16:", 1),
    ("e4m3 no subnormals", "vals.append(m * E4M3_SUBNORMAL_STEP)", "vals.append(0.0 if m else 0.0)", 1),
    ("ties away from zero", "((a - lo == hi - a) & (idx % 2 == 0))", "(a - lo == hi - a)", 1),
    ("ties to odd", "((a - lo == hi - a) & (idx % 2 == 0))", "((a - lo == hi - a) & (idx % 2 == 1))", 1),
    ("overflow to NaN instead of saturating", "return np.copysign(r, x)",
     "return np.copysign(np.where(np.abs(x) >= 464.0, np.nan, r), x)", 1),
    ("rotation signs ignored", "return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)",
     "return x @ hadamard(d) / np.sqrt(d)", 1),
    ("rotation not normalised", "return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)",
     "return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / d", 1),
    ("Hadamard block sign", "h = np.block([[h, h], [h, -h]])", "h = np.block([[h, h], [-h, h]])", 1),
    ("scale from the wrong maximum", "s = amax / E4M3_MAX if amax > 0.0 else 1.0",
     "s = amax / 240.0 if amax > 0.0 else 1.0", 1),
    ("one scale per tensor", "blk = x[t * block_rows:(t + 1) * block_rows]", "blk = x", 1),
    ("dequantise forgets the scale", "return codes * row_scale[:, None]", "return codes", 1),
    ("V rotated too", "for x in (qr, kr, np.asarray(v, dtype=np.float64)):",
     "for x in (qr, kr, rotate(v, signs)):", 1),
    ("only Q rotated", "kr = rotate(k, signs) if rotate_qk else", "kr = k if rotate_qk else", 1),
    ("P gain 32 instead of 64", "p_gain: float = 64.0", "p_gain: float = 32.0", 1),
    ("P gain 256 instead of 64", "p_gain: float = 64.0", "p_gain: float = 256.0", 1),
    ("P gain 16 instead of 64", "p_gain: float = 64.0", "p_gain: float = 16.0", 1),
    ("V-scale ratio inverted", "ratio = np.repeat(sv / sv.max(), block_rows)[:nk]",
     "ratio = np.repeat(sv.max() / sv, block_rows)[:nk]", 1),
    ("V-scale ratio against the smallest scale", "ratio = np.repeat(sv / sv.max(), block_rows)[:nk]",
     "ratio = np.repeat(sv / sv.min(), block_rows)[:nk]", 1),
    ("V-scale ratio dropped", "ratio = np.repeat(sv / sv.max(), block_rows)[:nk]",
     "ratio = np.repeat(sv / sv, block_rows)[:nk]", 1),
    ("P rounded without its gain", "pq = e4m3_round(p * p_gain * ratio[None, :]) / (p_gain * ratio[None, :])",
     "pq = e4m3_round(p * ratio[None, :]) / (ratio[None, :])", 1),
    ("rounded P used for l", "l = p.sum(axis=1)", "l = (e4m3_round(p * p_gain) / p_gain).sum(axis=1)", 1),
]


def _load_fp8_mutant(old, new, count):
    import oracle.attention as exact
    src = open(FP8_SRC, encoding="utf-8").read()
    assert src.count(old) >= count, f"mutation site not found: {old!r}"
    mutated = src.replace(old, new, count).replace("from .attention import naive_attention", "")
    mod = types.ModuleType("oracle_fp8_mutant")
    mod.__dict__["naive_attention"] = exact.naive_attention
    exec(compile(mutated, "oracle_fp8_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("name,old,new,count", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_mutant_is_caught(name, old, new, count):
    mod = _load_fp8_mutant(old, new, count)
    caught = []
    for pin in FP8_PINS:
        try:
            pin(mod)
        except Exception:  # noqa: BLE001 -- any failure of a pin counts
            caught.append(pin.__name__)
    assert caught, f"mutant '{name}' passed every pin"
