"""CPU tests of the fp64 oracle against its pins, plus mutation checks that a
plausible mistake anywhere in the oracle makes at least one pin fail."""
import os

import numpy as np
import pytest

import oracle
import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


# (text in fd_oracle.c, replacement, what the mistake is)
MUTATIONS = [
    ("const double ks = k_scale * scale_at(", "const double ks = 1.0 * scale_at(", "k_scale dropped"),
    ("s[t] = softmax_scale * dot;", "s[t] = dot;", "softmax_scale dropped"),
    ("const double vs = v_scale * scale_at(", "const double vs = 1.0 * scale_at(", "v_scale dropped"),
    ("o[d] += wt * (vs * vd);", "o[d] += s[t] * (vs * vd);", "weights not normalised"),
    ("*l = M + log(Z);", "*l = log(Z);", "lse misses the max"),
    ("*l = M + log(Z);", "*l = M + log(Z) / 2;", "lse wrong log"),
    ("int kvh = qh / group;", "int kvh = qh % num_kv_heads;", "GQA head map interleaved"),
    ("row = phys * page_size + t % page_size;", "row = phys * page_size + (t + 1) % page_size;",
     "page offset shifted"),
    ("int64_t phys = block_table[(int64_t)b * block_table_stride + t / page_size];",
     "int64_t phys = block_table[(int64_t)b * block_table_stride];", "always first page"),
    ("row = (int64_t)kv_start_idx[b] + t;", "row = (int64_t)kv_start_idx[b] + t + 1;",
     "contiguous row off by one"),
    ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);",
     "e4m3 bias"),
    ("mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);", "e4m3 subnormal"),
    ("else mag = ldexp(1.0 + (double)m / 128.0, e - 127);",
     "else mag = ldexp(1.0 + (double)m / 256.0, e - 127);", "bf16 mantissa"),
    ("for (int t = 0; t < T; ++t) { s[t] = exp(s[t] - M); Z += s[t]; }",
     "for (int t = 0; t < T; ++t) { s[t] = exp(s[t] - M); Z += s[t] * s[t]; }", "wrong sum"),
    ("size_t base = ((size_t)rows[t] * num_kv_heads + kvh) * head_dim;\n          const double vs",
     "size_t base = ((size_t)rows[t] * num_kv_heads + 0) * head_dim;\n          const double vs",
     "V read from head 0"),
    ("if (kind == FDO_SCALE_HEAD) return (double)arr[kvh];",
     "if (kind == FDO_SCALE_HEAD) return (double)arr[0];", "head scale of head 0"),
    ("if (kind == FDO_SCALE_TOKEN) return (double)arr[(size_t)row * num_kv_heads + kvh];",
     "if (kind == FDO_SCALE_TOKEN) return (double)arr[(size_t)kvh * num_kv_heads + row % num_kv_heads];",
     "token scale transposed"),
    ("scale_at(scale_kind, k_scales, rows[t], num_kv_heads, kvh)",
     "scale_at(scale_kind, k_scales, t, num_kv_heads, kvh)", "token scale by position"),
    ("scale_at(scale_kind, v_scales, rows[t], num_kv_heads, kvh)",
     "scale_at(scale_kind, k_scales, rows[t], num_kv_heads, kvh)", "V scaled by K scales"),
    ("if (v >= 128) v -= 256;", "if (v > 128) v -= 256;", "i8 code 0x80 read as +128"),
    ("  return (double)v;\n}", "  return (double)code;\n}", "i8 read as unsigned"),
    ("if (dtype == FDO_I8) return fdo_i8_value(", "if (dtype == FDO_I8) return fdo_e4m3_value(",
     "i8 cache decoded as e4m3"),
    ("if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {",
     "if (err < best_err) {", "e4m3 encoder ties to the lower code"),
    ("if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
     "if (f >= 0.5) r += 1.0;", "int8 encoder ties away from zero"),
    ("if (r > 127.0) r = 127.0;", "if (r > 128.0) r = 128.0;", "int8 encoder clamps at 128"),
    ("positions[b] + i, kv_rows);", "positions[b] + i + 1, kv_rows);", "append one token late"),
    ("          s = scale * scales[h];\n", "          s = scale;\n", "append ignores head scales"),
    ("(((size_t)b * n_new + i) * num_kv_heads + h) * head_dim;",
     "(((size_t)b * n_new + 0) * num_kv_heads + h) * head_dim;",
     "every new token takes the first token's rows"),
    ("          if (a > amax) amax = a;", "          if (a > amax && d == 0) amax = a;",
     "token scale from the first element"),
    ("        const float denom = qmax * scale;", "        const float denom = qmax;",
     "token scale ignores the per-tensor scale"),
    ("int T = seq_len[b] - (q_len - 1 - j);", "int T = seq_len[b] - (q_len - j);",
     "causal limit one key short"),
    ("int T = seq_len[b] - (q_len - 1 - j);", "int T = seq_len[b];",
     "new tokens see every key"),
    ("const size_t qi = ((size_t)b * num_q_heads + qh) * q_len + j;",
     "const size_t qi = ((size_t)b * num_q_heads + qh) * q_len + (q_len - 1 - j);",
     "query tokens reversed"),
    ("qv[d] = decode_elem(q, q_dtype, qi * head_dim + d);",
     "qv[d] = decode_elem(q, q_dtype, qi * head_dim + (head_dim - 1 - d));",
     "q transposed"),
]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[2] for m in MUTATIONS])
def test_mutated_oracle_fails_a_pin(tmp_path, mutation):
    old, new, what = mutation
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor missing: {what}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(orc)
        except (AssertionError, oracle.OracleError, FloatingPointError, ValueError):
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the mutation: {what}"


def test_golden_fixtures(orc):
    """The oracle reproduces its frozen fixtures (tests/golden) to 1e-12
    relative: guards against silent changes of its arithmetic and against a
    host whose libm rounds differently."""
    import importlib.util
    import json
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    for name, w, _ in mg.cases():
        doc = json.load(open(os.path.join(here, name)))
        ref_out = np.array([float.fromhex(x) for x in doc["out"]]).reshape(doc["out_shape"])
        ref_lse = np.array([float.fromhex(x) for x in doc["lse"]]).reshape(doc["lse_shape"])
        out, lse = orc.decode_attention(w)
        assert out.shape == ref_out.shape and lse.shape == ref_lse.shape, name
        assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-14), name
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse)) and np.array_equal(lse[~fin], ref_lse[~fin])
        assert np.allclose(lse[fin], ref_lse[fin], rtol=1e-12, atol=1e-14), name
