"""The oracle's pins fail on plausible mistakes planted in the oracle.

Each case copies oracle.c, plants one mistake in one function (a dropped
term, a wrong sign, index, position or order, a missing normalisation),
builds the copy into its own library under _build/, and runs the pin tests
(tests/test_oracle_pins.py) against it in a child process.  Mistakes in the
layer composition (oracle.py) go into a copy of the package, imported ahead
of the pins.  A case passes when the pins fail: exit status 1, a failed
assertion rather than a crash.  Unchanged copies taken the same routes pass.
The oracle's own files are never modified, and every planted mistake keeps
every memory access in bounds.
"""
import os
import subprocess
import sys

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "_build", "oracle_mutants")

# (name, the planted function's first line, text replaced, replacement)
MISTAKES = [
    ("rmsnorm sums instead of averaging", "void orc_rmsnorm(",
     "ss / (double)D + eps", "ss + eps"),
    ("rmsnorm ignores gamma", "void orc_rmsnorm(",
     "double g = gamma ? (double)gamma[d] : 1.0;", "double g = 1.0;"),
    ("rope rotates with the wrong sine sign", "void orc_rope(",
     "a * c - b * s", "a * c + b * s"),
    ("rope frequency exponent halved", "void orc_rope(",
     "-2.0 * (double)i / (double)r", "-1.0 * (double)i / (double)r"),
    ("rope rotates the first dims", "void orc_rope(",
     "int d0 = D - r;", "int d0 = 0;"),
    ("compressor window starts one stride early", "int orc_compress(",
     "int64_t u0 = (int64_t)m * (j + 1) - w;", "int64_t u0 = (int64_t)m * j - w;"),
    ("compressor weights not normalised", "int orc_compress(",
     "for (int s = 0; s < w; ++s) alpha[s] /= z;",
     "for (int s = 0; s < w; ++s) alpha[s] /= (z + 1.0);"),
    ("compressor ropes at the window's first token", "int orc_compress(",
     "orc_rope(acc, D, r, base, (int64_t)m * (j + 1) - 1, +1);",
     "orc_rope(acc, D, r, base, (int64_t)m * j, +1);"),
    ("compressor averages the indexer key", "int orc_compress(",
     "acc_i[d] += alpha[s] * orc_bf16_to_f64(irow[d]);",
     "acc_i[d] += orc_bf16_to_f64(irow[d]) / w;"),
    ("compressor ropes before the norm", "int orc_compress(",
     "            orc_rmsnorm(acc, D, gamma, eps);\n"
     "            orc_rope(acc, D, r, base, (int64_t)m * (j + 1) - 1, +1);",
     "            orc_rope(acc, D, r, base, (int64_t)m * (j + 1) - 1, +1);\n"
     "            orc_rmsnorm(acc, D, gamma, eps);"),
    ("compressor takes the previous token's gate", "int orc_compress(",
     "                double g = orc_bf16_to_f64(gate[(int64_t)b * L_cap + u]);\n"
     "                alpha[s]",
     "                double g = orc_bf16_to_f64(gate[(int64_t)b * L_cap + (u > 0 ? u - 1 : u)]);\n"
     "                alpha[s]"),
    ("hidden compressor shifts the key columns", "int orc_compress_hidden(",
     "memcpy(ik_out + o * dI, acc + D,", "memcpy(ik_out + o * dI, acc + D - 1,"),
    ("hidden compressor transposes W", "int orc_compress_hidden(",
     "for (int c = 0; c < P; ++c) proj[c] += xi * wr[c];",
     "for (int c = 0; c < P; ++c) proj[c] += xi * Wd[(int64_t)c * dm + i];"),
    ("hidden compressor norms one key column too", "int orc_compress_hidden(",
     "orc_rmsnorm(acc, D, gamma, eps);", "orc_rmsnorm(acc, D + (dI > 0 ? 1 : 0), gamma, eps);"),
    ("visibility off by one", "int64_t orc_visible(", "(t + 1) / m", "t / m"),
    ("indexer drops the ReLU", "int orc_indexer_scores(",
     "(dot > 0.0 ? dot : 0.0)", "dot"),
    ("indexer weight indexed by head only", "int orc_indexer_scores(",
     "(double)w[bt * HI + h]", "(double)w[h]"),
    ("top-k breaks ties to the larger index", "static int orc_pair_cmp(",
     "return (x->j < y->j) ? -1 : (x->j > y->j);",
     "return (x->j > y->j) ? -1 : (x->j < y->j);"),
    ("attention drops the logit scale", "static void attend(",
     "logit_buf[i] = scale * dot;", "logit_buf[i] = dot;"),
    ("attention lse drops the max", "static void attend(",
     "*lse = mx + log(z);", "*lse = log(z);"),
    ("HCA sees one entry too many", "int orc_attention(",
     "int64_t n = orc_visible(tp, m);", "int64_t n = orc_visible(tp + m, m);"),
    ("SWA window one token short", "int orc_attention(",
     "int64_t lo = tp - W + 1;", "int64_t lo = tp - W + 2;"),
    ("SWA keys not normalised", "int orc_attention(",
     "                    orc_rmsnorm(kr, D, gamma_kv, eps);\n", ""),
    ("SWA keys roped at the query's position", "int orc_attention(",
     "orc_rope(kr, D, r, base, u, +1);", "orc_rope(kr, D, r, base, tp, +1);"),
    ("queries not normalised", "static void prep_query(",
     "    orc_rmsnorm(out, D, gamma_q, eps);\n", ""),
    ("queries roped one position late", "static void prep_query(",
     "orc_rope(out, D, r, base, t, +1);", "orc_rope(out, D, r, base, t + 1, +1);"),
    ("merge leaves the sink out of Z", "int orc_merge(",
     "double z = sink ? exp((double)sink[h] - mx) : 0.0;", "double z = 0.0;"),
    ("merge rotates the output forward", "int orc_merge(",
     "orc_rope(y, D, r, base, pos[bt], -1);", "orc_rope(y, D, r, base, pos[bt], +1);"),
    ("merge returns the max as lse", "int orc_merge(",
     "lse_out[row] = lz;", "lse_out[row] = mx;"),
    ("sink weights leave the sink out of Z", "double orc_weights_with_sink(",
     "    double z = exp(sink - mx);\n", "    double z = 0.0;\n"),
    ("bf16 rounds ties away from zero", "uint16_t orc_f64_to_bf16(",
     "double r = nearbyint(scaled);", "double r = round(scaled);"),
    ("E4M3 subnormal spacing one step too fine", "uint8_t orc_f32_to_e4m3(",
     "if (q < -9) q = -9;", "if (q < -10) q = -10;"),
    ("E4M3 row scale inverted", "void orc_quantize_e4m3_row(",
     "*scale = amax / 448.0f;", "*scale = 448.0f / amax;"),
    ("MXFP4 scale exponent one too large", "static int orc_mx_scale_exp(",
     "int s = e - 1 - 2;", "int s = e - 2;"),
    ("MXFP4 nibbles swapped", "void orc_quantize_mxfp4_row(",
     "codes[i / 2] = (uint8_t)(lo | (hi << 4));", "codes[i / 2] = (uint8_t)(hi | (lo << 4));"),
    ("E2M1 rounds ties away from zero", "uint8_t orc_f64_to_e2m1(",
     "double v = ldexp(nearbyint(ldexp(a, -q)), q);", "double v = ldexp(round(ldexp(a, -q)), q);"),
    ("E2M1 does not saturate", "uint8_t orc_f64_to_e2m1(",
     "if (a >= 6.0) {", "if (a >= 8.0) {"),
    ("E2M1 exponent bias off by one", "double orc_e2m1_to_f64(",
     "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e - 2)"),
    ("MXFP4 element takes the neighbouring block's scale", "static double orc_mxfp4_value(",
     "orc_e8m0_to_f64(scales[d / 32])", "orc_e8m0_to_f64(scales[(d / 32) ^ 1])"),
    ("MXFP4 scores leave the query unquantised", "int orc_indexer_scores_mxfp4(",
     "qd[(size_t)h * dI + d] = orc_mxfp4_value(qc, qs, d);",
     "qd[(size_t)h * dI + d] = orc_bf16_to_f64(iq[(bt * HI + h) * dI + d]);"),
]


# Mistakes in the layer composition (oracle.py): how the branches are fed,
# kept and merged.
PY_MISTAKES = [
    ("merge leaves out the sink",
     'out, lse = merge(o_list, l_list, inp.get("sink"), pos, r, base)',
     'out, lse = merge(o_list, l_list, None, pos, r, base)'),
    ("merge rotates back by the next position",
     'out, lse = merge(o_list, l_list, inp.get("sink"), pos, r, base)',
     'out, lse = merge(o_list, l_list, inp.get("sink"), pos + 1, r, base)'),
    ("the HCA branch is not merged",
     "        o_list.append(o)\n        l_list.append(l)\n        if keep:\n"
     "            res.update(kv_h=kv_h",
     "        if keep:\n            res.update(kv_h=kv_h"),
    ("the CSA cache is built one entry short",
     "n = min(L // m, visible(tmax, m)) if L >= m else 0",
     "n = min(L // m, visible(tmax, m)) - 1 if L >= m else 0"),
    ("the indexer scores with the wrong stride",
     'scores = indexer_scores(inp["iq"], inp["w"], ik_c, pos, m)',
     'scores = indexer_scores(inp["iq"], inp["w"], ik_c, pos, m + 1)'),
    ("the SWA window is halved",
     'attention(KIND_SWA, inp["q"], kv_raw, pos, W=cfg["W"]',
     'attention(KIND_SWA, inp["q"], kv_raw, pos, W=cfg["W"] // 2'),
]


@pytest.fixture(scope="module", autouse=True)
def _clean_up_builds():
    """The planted builds live only while this module runs."""
    import shutil
    yield
    shutil.rmtree(OUT, ignore_errors=True)


def _function(text, first_line):
    a = text.index(first_line)
    return a, text.index("\n}\n", a) + 3


def _pins_against(source, tag):
    """Build `source` as its own oracle library and run the pins on it."""
    os.makedirs(OUT, exist_ok=True)
    c_path = os.path.join(OUT, tag + ".c")
    with open(c_path, "w") as f:
        f.write(source)
    lib = obuild.compile_library(c_path, os.path.join(OUT, tag + ".so"))
    env = dict(os.environ, ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unchanged_copy_passes_the_pins():
    """The control: the same route with nothing planted passes, so a planted
    case fails because of its mistake and not because of the route."""
    r = _pins_against(open(obuild.SRC).read(), "control")
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,fn,old,new", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_pins_fail_on_planted_mistake(name, fn, old, new):
    src = open(obuild.SRC).read()
    a, b = _function(src, fn)
    body = src[a:b]
    assert body.count(old) == 1, f"the text to replace must occur once in {fn}"
    tag = "m%02d" % [m[0] for m in MISTAKES].index(name)
    r = _pins_against(src[:a] + body.replace(old, new) + src[b:], tag)
    assert r.returncode == 1, (r.returncode, r.stdout[-2000:])
    assert "failed" in r.stdout.splitlines()[-1]



def _package_copy(tag, oracle_py):
    """A copy of the oracle package under _build/ with the given oracle.py."""
    import shutil
    pkg = os.path.join(OUT, tag, "oracle")
    os.makedirs(pkg, exist_ok=True)
    for f in ("__init__.py", "build.py"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(pkg, f))
    with open(os.path.join(pkg, "oracle.py"), "w") as f:
        f.write(oracle_py)
    return pkg


def _pins_with_package(pkg):
    """Run the pins in a child that imports the package copy first (the
    unchanged C library underneath)."""
    driver = ("import sys; sys.path.insert(0, %r); import oracle; "
              "assert oracle.__file__.startswith(%r); import pytest; "
              "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', %r]))"
              % (os.path.dirname(pkg), pkg, os.path.join(ROOT, "tests", "test_oracle_pins.py")))
    return subprocess.run([sys.executable, "-c", driver], cwd=ROOT, capture_output=True,
                          text=True, env=dict(os.environ, ORACLE_LIB=obuild.build()),
                          timeout=600)


def test_unchanged_package_copy_passes_the_pins():
    """The control of the composition cases."""
    src = open(os.path.join(ROOT, "oracle", "oracle.py")).read()
    r = _pins_with_package(_package_copy("pycontrol", src))
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-2000:])


@pytest.mark.parametrize("name,old,new", PY_MISTAKES, ids=[m[0] for m in PY_MISTAKES])
def test_pins_fail_on_planted_composition_mistake(name, old, new):
    """A copy of the oracle package with one mistake in oracle.py is imported
    ahead of the pins."""
    src = open(os.path.join(ROOT, "oracle", "oracle.py")).read()
    assert src.count(old) == 1
    tag = "py%02d" % [m[0] for m in PY_MISTAKES].index(name)
    r = _pins_with_package(_package_copy(tag, src.replace(old, new)))
    assert r.returncode == 1, (r.returncode, r.stdout[-2000:], r.stderr[-2000:])
    assert "failed" in r.stdout.splitlines()[-1]
