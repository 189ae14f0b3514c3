"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is a copy of ``oracle/zero_oracle.cpp`` with one plausible mistake
(a dropped term, a wrong sign, a swapped operand, an off-by-one ...), compiled
on the CPU into a temporary directory.  The test requires that at least one
pin in ``oracle_pins`` fails on every mutant, so that the pins really fix each
part of the oracle.  Nothing here touches a GPU.
"""
import concurrent.futures as cf
import os
import tempfile

import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("m EMA drops (1-beta1)", "mj = d->b1 * mj + d->omb1 * g;", "mj = d->b1 * mj + g;"),
    ("v uses g not g*g", "d->omb2 * (g * g)", "d->omb2 * g"),
    ("beta1 used for v", "vj = d->b2 * vj", "vj = d->b1 * vj"),
    ("eps inside the root", "std::sqrt(vj) * d->isb2 + d->eps", "std::sqrt(vj + d->eps) * d->isb2"),
    ("update sign flipped", "pj = pj - d->step_size * (mj / den);", "pj = pj + d->step_size * (mj / den);"),
    ("decay after the Adam term",
     "pj = pj * d->decay;\n    pj = pj - d->step_size * (mj / den);",
     "pj = pj - d->step_size * (mj / den);\n    pj = pj * d->decay;"),
    ("decay dropped", "pj = pj * d->decay;", ""),
    ("bias correction exponent t+1", "std::pow(hp->beta1, t)", "std::pow(hp->beta1, t + 1.0)"),
    ("step size ignores bc1", "d->step_size = (float)(lr / bc1);", "d->step_size = (float)(lr);"),
    ("isb2 inverted", "(float)(1.0 / std::sqrt(bc2))", "(float)(std::sqrt(bc2))"),
    ("t advances on skipped steps", "st->skipped_total += 1;", "st->skipped_total += 1; st->t += 1;"),
    ("scale grows on overflow", "(double)scale / hp->scale_factor", "(double)scale * hp->scale_factor"),
    ("clean counter kept on overflow", "st->clean = 0;\n    st->skipped_total", "st->skipped_total"),
    ("min scale floor dropped", "if (lowered < hp->min_scale) lowered = hp->min_scale;", ""),
    ("window off by one", "st->clean == hp->scale_window", "st->clean > hp->scale_window"),
    ("clip clamps the wrong way", "if (clip > 1.0) clip = 1.0;", "if (clip < 1.0) clip = 1.0;"),
    ("norm not unscaled", "std::sqrt(global.sumsq) * inv", "std::sqrt(global.sumsq)"),
    ("unscale forgets the divisor", "1.0 / ((double)scale * divisor)", "1.0 / ((double)scale)"),
    ("reduce drops the last buffer", "for (int32_t b = 0; b < nbuf; ++b)", "for (int32_t b = 0; b + 1 < nbuf; ++b)"),
    ("reduce in reverse order", "acc = acc + orc_16_to_f32(bufs[b][j], dtype);",
     "acc = acc + orc_16_to_f32(bufs[nbuf - 1 - b][j], dtype);"),
    ("NaN not treated as overflow", "if (!std::isfinite(s[j])) st.nonfinite = 1;", "if (std::isinf(s[j])) st.nonfinite = 1;"),
    ("fold drops the overflow flag", "if (per_rank[r].nonfinite) st.nonfinite = 1;", ""),
    ("fp16 ties round down", "if (rem > half || (rem == half && (n & 1u))) n += 1;", "if (rem > half) n += 1;"),
    ("subnormal decode off by 2x", "std::ldexp((double)man, 1 - bias - mbits)", "std::ldexp((double)man, -bias - mbits)"),
    ("bf16 mantissa width", "*mbits = 7; *ebits = 8;", "*mbits = 8; *ebits = 7;"),
    ("shards not padded", "int64_t shard = (numel + world - 1) / world;", "int64_t shard = numel / world;"),
    ("stage 2 keeps full gradients", "case 2: return 2 * psi + 2 * s + 12 * s;", "case 2: return 2 * psi + 2 * psi + 12 * s;"),
    ("hysteresis ignored", "if (st->overflows >= hp->hysteresis) {", "if (st->overflows >= 1) {"),
    ("warm-up one update late", "const double frac = t < (double)hp->warmup_num_steps ? t / (double)hp->warmup_num_steps : 1.0;",
     "const double frac = t - 1.0 < (double)hp->warmup_num_steps ? (t - 1.0) / (double)hp->warmup_num_steps : 1.0;"),
    ("growth keeps the overflow count", "    st->clean = 0;\n    st->overflows = 0;\n  }", "    st->clean = 0;\n  }"),
    ("16-bit copy in the other format", "p16[j] = orc_f32_to_16(pj, pdtype);",
     "p16[j] = orc_f32_to_16(pj, 1 - pdtype);"),
    ("low-precision master widened from the other format",
     "float pj = master ? master[j] : orc_16_to_f32(p16[j], pdtype);",
     "float pj = master ? master[j] : orc_16_to_f32(p16[j], 1 - pdtype);"),
    ("low-precision master starts from zero",
     "float pj = master ? master[j] : orc_16_to_f32(p16[j], pdtype);",
     "float pj = master ? master[j] : 0.0f;"),
]


def _build(idx, src_text, tmpdir):
    name, old, new = MUTANTS[idx]
    assert src_text.count(old) >= 1, f"mutant pattern not found: {name}"
    text = src_text.replace(old, new, 1)
    path = os.path.join(tmpdir, f"mut{idx}.cpp")
    with open(path, "w") as f:
        f.write(text)
    return oracle.compile_source(path, os.path.join(tmpdir, f"libmut{idx}.so"))


@pytest.fixture(scope="module")
def mutant_libs():
    src = open(oracle.SOURCE).read()
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        paths = list(ex.map(lambda i: _build(i, src, tmp), range(len(MUTANTS))))
    return paths


def _caught(orc):
    # cheap pins first; the cast sweeps last
    pins = sorted(oracle_pins.PINS, key=lambda f: "cast" in f.__name__)
    for pin in pins:
        try:
            pin(orc)
        except Exception as e:  # any failure of a pin counts as caught
            return pin.__name__, repr(e)[:120]
    return None


@pytest.mark.parametrize("idx", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(mutant_libs, idx):
    orc = oracle.Oracle(mutant_libs[idx])
    caught = _caught(orc)
    assert caught is not None, f"no pin detects the planted mistake: {MUTANTS[idx][0]}"


def test_sum_of_squares_compensation_mutant_is_caught(tmp_path):
    """Dropping the compensation (plain sequential binary64 summation) is
    caught by the correctly-rounded pin."""
    src = open(oracle.SOURCE).read()
    old = "st.sumsq = sum + comp;"
    assert src.count(old) == 1
    path = tmp_path / "mut_sumsq.cpp"
    path.write_text(src.replace(old, "st.sumsq = sum;"))
    lib = oracle.compile_source(str(path), str(tmp_path / "libmuts.so"))
    assert _caught(oracle.Oracle(lib)) is not None


def test_consolidation_mutant_is_caught(tmp_path):
    src = open(oracle.SOURCE).read()
    old = "for (int64_t j = b[0]; j < b[1]; ++j) out[j] = shard_master[r][j - b[0]];"
    new = ("for (int64_t j = b[0]; j < b[1]; ++j) "
           "out[j] = shard_master[r][j - b[0] + (j + 1 < b[1] ? 1 : 0)];")
    assert src.count(old) == 1
    path = tmp_path / "mut_consolidate.cpp"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / "libmutc.so"))
    assert _caught(oracle.Oracle(lib)) is not None
