"""The pins must be able to fail: each case below plants one plausible mistake
(a dropped term, a wrong sign, bias, index, stride or rounding rule) in a copy
of the C oracle, and the CPU pins of tests/test_oracle_pins.py, run against
that copy, must report at least one failure.  Runs on the CPU only; the copies
live in a temporary directory."""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in oracle/dsv4_oracle.c, planted replacement)
MUTANTS = [
    # number formats
    ("e4m3 ties away from zero", "double n = nearbyint(ldexp(a, -qexp));",
     "double n = round(ldexp(a, -qexp));"),
    ("e4m3 saturates to NaN", "if (a >= E4M3_MAX) return sign | 0x7E;",
     "if (a >= E4M3_MAX) return sign | 0x7F;"),
    ("e4m3 subnormal step", "int qexp = (E >= 1) ? (e - 1) - 3 : -9;",
     "int qexp = (E >= 1) ? (e - 1) - 3 : -10;"),
    ("e4m3 decode bias", "else v = ldexp(8.0 + M, E - 10);", "else v = ldexp(8.0 + M, E - 9);"),
    ("bf16 truncates", "double r = ldexp(nearbyint(ldexp(ax, -qexp)), qexp);",
     "double r = ldexp(floor(ldexp(ax, -qexp)), qexp);"),
    ("scale bound strict", "while (!(a <= ldexp(E4M3_MAX, e))) e++;",
     "while (!(a < ldexp(E4M3_MAX, e))) e++;"),
    ("amax floor", "#define AMAX_FLOOR 1e-4f", "#define AMAX_FLOOR 1e-6f"),
    # inverse rotation
    ("rotation: y1 sign", "*y1 = fmaf(b, c, -as);", "*y1 = fmaf(b, c, as);"),
    ("rotation: forward y0", "*y0 = fmaf(a, c, bs);", "*y0 = fmaf(a, c, -bs);"),
    ("rotation: dropped term", "*y0 = fmaf(a, c, bs);", "*y0 = a * c;"),
    ("rotation: cos and sin swapped",
     "oracle_inv_rope_pair(a, b, crow[i], crow[half + i],",
     "oracle_inv_rope_pair(a, b, crow[half + i], crow[i],"),
    ("rotation: half-split pairs",
     "float a = dst[nope_dim + 2 * i], b = dst[nope_dim + 2 * i + 1];",
     "float a = dst[nope_dim + i], b = dst[nope_dim + half + i];"),
    ("rotation: position ignored",
     "float* y = (float*)malloc(sizeof(float) * (size_t)D);\n"
     "        const float* crow = cache + positions[t] * rope_dim;",
     "float* y = (float*)malloc(sizeof(float) * (size_t)D);\n"
     "        const float* crow = cache + (t % max_pos) * rope_dim;"),
    # block quantisation and layout
    ("scale byte bias", "uint32_t byte = (uint32_t)(e + 127);",
     "uint32_t byte = (uint32_t)(e + 128);"),
    ("scale applied with the wrong sign",
     "double q = ldexp((double)y[kb * quant_group_size + j], -e);",
     "double q = ldexp((double)y[kb * quant_group_size + j], e);"),
    ("amax over block 0 only", "float v = fabsf(y[kb * quant_group_size + j]);",
     "float v = fabsf(y[j]);"),
    ("amax without abs", "float v = fabsf(y[kb * quant_group_size + j]);",
     "float v = y[kb * quant_group_size + j];"),
    ("packed byte order", "packed[kb / 4] |= byte << (8 * (kb % 4));",
     "packed[kb / 4] |= byte << (8 * (3 - kb % 4));"),
    ("codes token-major", "uint8_t* qrow = out_fp8 + (g * T + t) * D;",
     "uint8_t* qrow = out_fp8 + (t * n_groups + g) * D;"),
    ("scales pack-major", "out_scale[(g * PK + p) * T_al + t] = (int32_t)packed[p];",
     "out_scale[(p * n_groups + g) * T_al + t] = (int32_t)packed[p];"),
    ("TMA alignment of 8 bytes", "const int64_t per16 = 16 / 4;",
     "const int64_t per16 = 16 / 2;"),
    # grouped GEMM
    ("GEMM: group rows dropped", "const int64_t row = g * R + n;", "const int64_t row = n;"),
    ("GEMM: activation scale word",
     "uint32_t word = (uint32_t)x_scale[(g * PK + kb / 4) * T_al + t];",
     "uint32_t word = (uint32_t)x_scale[(g * PK + kb % PK) * T_al + t];"),
    ("GEMM: activation scale bias", "int e = (int)((word >> (8 * (kb % 4))) & 0xFF) - 127;",
     "int e = (int)((word >> (8 * (kb % 4))) & 0xFF) - 128;"),
    ("GEMM: weight scale row block", "const uint8_t* srow = w_scale + (row / 128) * KB;",
     "const uint8_t* srow = w_scale + (n / 128) * KB;"),
    ("GEMM: weight scale dropped", "acc += xs[k] * (lut[wrow[k]] * sc);",
     "acc += xs[k] * lut[wrow[k]];"),
    # z re-quantisation
    ("re-quant amax without abs", "float v = fabsf(oracle_bf16_to_float(src[j]));",
     "float v = oracle_bf16_to_float(src[j]);"),
    ("re-quant scale byte",
     "out_scale[(kb / 4) * T_al + t] |= (int32_t)((uint32_t)(e + 127) << (8 * (kb % 4)));",
     "out_scale[(kb / 4) * T_al + t] |= (int32_t)((uint32_t)(e + 126) << (8 * (kb % 4)));"),
    # bf16 variants
    ("bf16: nope lanes zeroed", "for (int64_t j = 0; j < nope_dim; j++) dst[j] = src[j];",
     "for (int64_t j = 0; j < nope_dim; j++) dst[j] = 0;"),
    ("bf16 GEMM: group rows dropped", "const uint16_t* wr = w_bf16 + (g * R + n) * D;",
     "const uint16_t* wr = w_bf16 + n * D;"),
]


def _run_pins_on(i, name, text, planted, src, base):
    d = os.path.join(base, f"mutant{i}")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(d, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    with open(os.path.join(d, "oracle", "dsv4_oracle.c"), "w") as f:
        f.write(src.replace(text, planted))
    env = dict(os.environ, PYTHONPATH=d + os.pathsep + ROOT, OMP_NUM_THREADS="1")
    # the planted copy must build (a compile error is not a caught mistake)
    b = subprocess.run([sys.executable, "-c", "import oracle; oracle.build()"], cwd=d, env=env,
                       capture_output=True, text=True, timeout=300)
    if b.returncode != 0:
        return name, -1
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=d, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_planted_mistake_fails_a_pin(tmp_path):
    with open(os.path.join(ROOT, "oracle", "dsv4_oracle.c")) as f:
        src = f.read()
    for name, text, _ in MUTANTS:
        assert src.count(text) == 1, f"{name}: the oracle text it mutates changed"
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(lambda im: _run_pins_on(im[0], *im[1], src, str(tmp_path)),
                              enumerate(MUTANTS)))
    survivors = [name for name, rc in results if rc == 0]
    errors = [name for name, rc in results if rc not in (0, 1)]
    assert not errors, f"the planted copy did not build, or the pins did not run, for: {errors}"
    assert not survivors, f"no pin fails for: {survivors}"
