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
    "key_reads_value_half": ("return orc_e4m3(row[d]) * p->k_scale;",
                             "return orc_e4m3(row[ORC_D + d]) * p->k_scale;"),
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


# The prefill routines compose the decode routines per request in Python
# (oracle/__init__.py); their plausible mistakes are planted in a copy of that
# module, which a child process loads as `oracle` before running the prefill
# pins against the unmodified C library.
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")
PY_MUTANTS = {
    "unmodified": None,
    # the chunk placed at the start of its sequence instead of its end
    "prefill_tokens_at_sequence_start": (
        "np.asarray(seq_lens)[b:b + 1], n,",
        "np.minimum(np.asarray(seq_lens)[b:b + 1], n), n,"),
    # a request's queries taken in reverse token order
    "prefill_query_rows_reversed": (
        "p = Problem(q_bits[s:s + n], kv,",
        "p = Problem(np.ascontiguousarray(q_bits[s:s + n][::-1]), kv,"),
    # the selection made as if the chunk started the sequence
    "prefill_selection_at_sequence_start": (
        "np.asarray(seq_lens, dtype=np.int32)[b:b + 1],\n                            n, k)",
        "np.minimum(np.asarray(seq_lens, dtype=np.int32)[b:b + 1], n),\n"
        "                            n, k)"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_prefill_mutant_is_caught(name, tmp_path):
    import oracle
    src = open(PY_SRC).read()
    if PY_MUTANTS[name] is not None:
        old, new = PY_MUTANTS[name]
        assert src.count(old) == 1, f"mutation site for {name} not found"
        src = src.replace(old, new)
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src)
    script = (
        "import importlib.util, sys\n"
        f"spec = importlib.util.spec_from_file_location('oracle', {str(pkg / '__init__.py')!r},\n"
        f"    submodule_search_locations=[{str(pkg)!r}])\n"
        "m = importlib.util.module_from_spec(spec)\n"
        "sys.modules['oracle'] = m\n"
        "spec.loader.exec_module(m)\n"
        "import pytest\n"
        "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', '-k', 'prefill',\n"
        f"    {os.path.join(ROOT, 'tests', 'test_oracle_pins.py')!r}]))\n")
    env = dict(os.environ, MSA_ORACLE_LIB=oracle.build())
    r = subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    if PY_MUTANTS[name] is None:     # the harness itself: an unmodified copy passes every pin
        assert r.returncode == 0, r.stdout[-2000:]
    else:                            # a pin fails (exit status 1), not the harness
        assert r.returncode == 1, f"mutant {name}: status {r.returncode}\n{r.stdout[-2000:]}"
