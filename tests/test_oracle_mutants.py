"""Each plausible mistake planted in a copy of the oracle must make at least
one pin fail.  The mutants are compiled from the oracle source with one
substitution each and run in a child process through the pin tests."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "msa_oracle.c")

MUTANTS = {
    "group_mapping_modulo": ("int g = h / G;\n    int64_t pos", "int g = h % p->Hkv;\n    int64_t pos"),
    "causal_offset_off_by_one": ("return (int64_t)p->seq_lens[b] - p->Q + j;",
                                 "return (int64_t)p->seq_lens[b] - p->Q + j + 1;"),
    "value_reads_key_half": ("return orc_e4m3(row[ORC_D + d]) * p->v_scale;",
                             "return orc_e4m3(row[d]) * p->v_scale;"),
    "value_scale_dropped": ("return orc_e4m3(row[ORC_D + d]) * p->v_scale;",
                            "return orc_e4m3(row[ORC_D + d]);"),
    "key_scale_dropped": ("return orc_e4m3(row[d]) * p->k_scale;", "return orc_e4m3(row[d]);"),
    "sm_scale_dropped": ("return p->sm_scale * acc;", "return acc;"),
    "ties_to_higher_index": ("return (x->block < y->block) ? -1 : (x->block > y->block) ? 1 : 0;",
                             "return (x->block < y->block) ? 1 : (x->block > y->block) ? -1 : 0;"),
    "score_causal_mask_strict": ("if (n * ORC_PAGE + t > pos)\n                        break;",
                                 "if (n * ORC_PAGE + t >= pos)\n                        break;"),
    "attend_mask_dropped": ("for (int t = 0; t < ORC_PAGE && (int64_t)n * ORC_PAGE + t <= pos; ++t) {\n            double w",
                            "for (int t = 0; t < ORC_PAGE; ++t) {\n            double w"),
    "current_block_not_forced": ("kept[n_kept++] = cur;\n                    qsort",
                                 "kept[n_kept++] = cand[k - 1].block;\n                    qsort"),
    "output_not_sorted": ("qsort(kept, (size_t)n_kept, sizeof(int64_t), orc_int64_ascending);", ";"),
    "subnormal_exponent": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "combine_weight_inverted": ("double w = exp2(m - M);", "double w = exp2(M - m);"),
    "score_max_over_one_head": ("for (int hh = 0; hh < G; ++hh) {", "for (int hh = 0; hh < 1; ++hh) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))     # every copy of the site gets the same mistake
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-shared", "-fPIC", "-pthread", str(mut),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, MSA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
