"""Pins of the oracle's cache-format quantizers: hand-worked examples, entry
sizes printed on the pages, and the defining nearest-value properties checked
with numpy and torch (independent of the oracle's code)."""
import json

import numpy as np
import torch

from conftest import golden_path, read_table

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nib(codes: np.ndarray) -> np.ndarray:
    """[n, B] bytes -> [n, 2B] 4-bit codes, element 2i from the low nibble."""
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


def _val(c: np.ndarray) -> np.ndarray:
    v = E2M1[c & 7]
    return np.where(c & 8, -v, v)


def test_entry_sizes(oracle_mod):
    tab = {k: v for k, v in read_table("bytes_per_token.txt")}
    c, s = oracle_mod.quantize_main(np.zeros((1, 512), np.float32))
    c2, s2 = oracle_mod.quantize_index(np.zeros((1, 128), np.float32))
    assert c.nbytes + s.nbytes == int(tab["main_entry_bytes"])
    assert c2.nbytes + s2.nbytes == int(tab["index_entry_bytes"])
    assert c.nbytes + s.nbytes + c2.nbytes + s2.nbytes == int(tab["entry_bytes"])


def test_worked_examples(oracle_mod):
    ex = json.load(open(golden_path("quantizer_examples.json")))
    for e in ex["main"]:
        x = np.zeros((1, 512), np.float32)
        x[0, :16] = e["x"]
        c, s = oracle_mod.quantize_main(x)
        assert s[0, 0] == e["scale"], e["why"]
        assert list(c[0, :8]) == e["codes"], e["why"]
        assert np.all(s[0, 1:] == 0) and np.all(c[0, 8:] == 0)
    for e in ex["index"]:
        x = np.zeros((1, 128), np.float32)
        x[0, :len(e["x_head"])] = e["x_head"]
        c, s = oracle_mod.quantize_index(x)
        assert s[0, 0] == e["scale"], e["why"]
        assert list(c[0, :len(e["codes_head"])]) == e["codes_head"], e["why"]


def test_main_quantizer_properties(oracle_mod):
    """Scale byte = torch's nearest-even E4M3 of fp32(amax/6); each code is a
    nearest E2M1 of fp32(x/s) with even ties; zero scale gives zero codes."""
    rng = np.random.default_rng(1)
    parts = [rng.standard_normal((256, 512)),
             rng.standard_normal((64, 512)) * 1e-3,
             rng.standard_normal((64, 512)) * 300.0,
             np.repeat(rng.integers(-12, 13, (64, 512)) / 4.0, 1, axis=0)]
    x = np.concatenate(parts).astype(np.float32)
    x[3, 16:32] = 0.0
    x[4, 32:48] = -1e-9
    c, s = oracle_mod.quantize_main(x)
    g = np.abs(x).reshape(-1, 32, 16).max(-1)
    t = (g.astype(np.float32) / np.float32(6.0)).astype(np.float32)
    ref_s = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref_s, s)
    sv = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    codes = _nib(c).reshape(-1, 32, 16)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = (x.reshape(-1, 32, 16) / sv[..., None]).astype(np.float32).astype(np.float64)
    nz = sv[..., None].repeat(16, -1) != 0
    err = np.abs(y - _val(codes))
    for alt in range(8):
        cand = np.abs(np.abs(y) - E2M1[alt])
        assert np.all(err[nz] <= cand[nz] + 0.0)
    assert np.all(codes[~nz] == 0)
    # signs follow x wherever the magnitude is nonzero
    nzc = (codes & 7) != 0
    assert np.all(((codes & 8) != 0)[nzc] == (x.reshape(-1, 32, 16) < 0)[nzc])


def test_index_quantizer_properties(oracle_mod):
    """Scale = 2^(floor(log2 amax) - 2) (OCP MX); codes nearest E2M1 of x / scale."""
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal((256, 128)), rng.standard_normal((32, 128)) * 1e-30,
                        rng.standard_normal((32, 128)) * 1e30]).astype(np.float32)
    c, s = oracle_mod.quantize_index(x)
    amax = np.abs(x).reshape(-1, 4, 32).max(-1).astype(np.float64)
    e = np.floor(np.log2(amax)).astype(np.int64) - 2
    assert np.array_equal(np.clip(e, -127, 127) + 127, s.astype(np.int64))
    X = np.exp2(s.astype(np.float64) - 127)
    y = x.reshape(-1, 4, 32) / X[..., None]
    codes = _nib(c).reshape(-1, 4, 32)
    err = np.abs(y - _val(codes))
    for alt in range(8):
        assert np.all(err <= np.abs(np.abs(y) - E2M1[alt]))
    # values in (6, 8) * X clip to 6 * X: the OCP rule's known saturation
    assert np.all(np.abs(_val(codes)) <= 6)


def test_dequant_roundtrip(oracle_mod):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((32, 512)).astype(np.float32)
    c, s = oracle_mod.quantize_main(x)
    d = oracle_mod.dequant_main(c, s)
    sv = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(d.reshape(-1, 32, 16), _val(_nib(c).reshape(-1, 32, 16)) * sv[..., None])
    # re-quantizing the dequantized values is a fixed point when no scale saturates
    c2, s2 = oracle_mod.quantize_main(d.astype(np.float32))
    assert np.array_equal(oracle_mod.dequant_main(c2, s2), d)
    k = rng.standard_normal((32, 128)).astype(np.float32)
    ci, si = oracle_mod.quantize_index(k)
    di = oracle_mod.dequant_index(ci, si)
    assert np.array_equal(di.reshape(-1, 4, 32),
                          _val(_nib(ci).reshape(-1, 4, 32)) * np.exp2(si.astype(float) - 127)[..., None])


def test_margins_flag_decision_points(oracle_mod):
    x = np.zeros(16)
    x[0] = 6.0 * 1.6875  # amax/6 exactly on the E4M3 midpoint between 1.625 and 1.75
    assert oracle_mod.main_group_margins(x)[0] == 0.0
    x = np.zeros(32)
    x[0] = 4.0  # amax exactly a power of two
    assert oracle_mod.index_group_margins(x)[0] == 0.0
    x[0] = 3.0
    x[1] = 0.25 * 0.5 * 1.0000001  # element near the 0/0.5 midpoint at X = 0.5
    assert oracle_mod.index_group_margins(x)[0] < 1e-6
