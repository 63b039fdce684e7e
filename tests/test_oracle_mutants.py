"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a temporary copy of the oracle's C source,
builds it with gcc, and checks that at least one pin (golden traces, the
recency-list model, invariants, closed forms) rejects the planted oracle.
The oracle in the repository is never modified.
"""

import os
import subprocess
import sys

import pytest

import oracle as O
from golden_trace import names
import test_oracle as T
import test_oracle_paged as TP

SRC = os.path.join(os.path.dirname(O.__file__), "hisparse_oracle.c")

# (id, original text, planted mistake)
MUTANTS = [
    ("lru_newest_first",
     "return x->last_used < y->last_used ? -1 : 1;",
     "return x->last_used < y->last_used ? 1 : -1;"),
    ("slot_tiebreak_reversed",
     "return (x->slot > y->slot) - (x->slot < y->slot);",
     "return (x->slot < y->slot) - (x->slot > y->slot);"),
    ("misses_not_sorted",
     "qsort(miss, (size_t)m, sizeof(int32_t), cmp_i32);",
     ";"),
    ("evicted_token_not_unmapped",
     "if (s2t[v] >= 0) t2s[s2t[v]] = -1;",
     ";"),
    ("hits_not_stamped",
     "lu[t2s[t]] = tick;",
     "if (!is_hit_slot[t2s[t]]) lu[t2s[t]] = tick;"),
    ("hit_slots_evictable",
     "if (!is_hit_slot[s]) { cand[nc]",
     "if (1) { cand[nc]"),
    ("fast_path_strict",
     "if (S <= D) {\n        for (int j = 0; j < k; ++j)\n            if (!done[j]) out[j] = topk[j];",
     "if (S < D) {\n        for (int j = 0; j < k; ++j)\n            if (!done[j]) out[j] = topk[j];"),
    ("prefill_oldest_tokens",
     "s2t[i] = S - n + i;\n                    t2s[S - n + i] = i;",
     "s2t[i] = i;\n                    t2s[i] = i;"),
    ("tick_not_advanced",
     "uint32_t tick = ++o->tick[layer][r];",
     "uint32_t tick = o->tick[layer][r] + 1;"),
    ("copy_transposed",
     "copy_row(o, a, r, t, v);",
     "copy_row(o, a, r, v, t);"),
    ("plan_transposed",
     "plan[2 * i] = plan_host_slot(o, r, t);\n        plan[2 * i + 1] = v;",
     "plan[2 * i] = v;\n        plan[2 * i + 1] = plan_host_slot(o, r, t);"),
    ("duplicates_accepted",
     "if (v[i] == v[i - 1]) { st = HSO_DUPLICATE; break; }",
     ";"),
    ("error_keeps_outputs",
     "for (int j = 0; j < k; ++j) out[j] = -1;\n        return;",
     "return;"),
    ("backup_skips_device",
     "memcpy(hso_dev_row(o, layer, r, p), rows + (int64_t)r * o->B, (size_t)o->B);",
     ";"),
    ("replay_wrong_layer",
     "memcpy(hso_dev_row(o, layer, r, v), o->host[layer] + row * o->B, (size_t)o->B);",
     "memcpy(hso_dev_row(o, 0, r, v), o->host[layer] + row * o->B, (size_t)o->B);"),
    ("resident_after_hot",
     "        if (row >= 0) {\n            out[j] = (int32_t)(HSO_RESIDENT_FLAG | row);",
     "        if (row >= 0 && (S <= D || o->tok2slot[a][o->host_off[r] + topk[j]] < 0)) {\n"
     "            out[j] = (int32_t)(HSO_RESIDENT_FLAG | row);"),
    ("resident_hits_stamped",
     "        if (done[j]) continue;\n        if (t < 0) { out[j] = -1; continue; }",
     "        if (done[j]) { if (t2s[t] >= 0) lu[t2s[t]] = tick; continue; }\n"
     "        if (t < 0) { out[j] = -1; continue; }"),
    ("resident_counted_as_miss",
     "        if (t < 0 || done[j]) continue;",
     "        if (t < 0) continue;"),
    ("resident_row_offset_dropped",
     "return (int64_t)rt->blocks[b] * rt->block_size + t % rt->block_size;",
     "return (int64_t)rt->blocks[b] * rt->block_size;"),
    ("paged_row_offset_dropped",
     "return (int64_t)id * o->hb + t % o->hb;",
     "return (int64_t)id * o->hb;"),
    ("paged_highest_free_first",
     "int32_t id = 0;\n            while (o->in_use[id]) ++id;",
     "int32_t id = o->pool_blocks - 1;\n            while (o->in_use[id]) --id;"),
    ("paged_partial_reservation",
     "    if (need > hso_free_blocks(o)) return -2;\n",
     ""),
    ("paged_release_keeps_blocks",
     "            o->in_use[o->blocks[r][b]] = 0;\n",
     ""),
    ("paged_plan_records_token",
     "return o->hb == 0 ? t : (int32_t)host_row_of(o, r, t);",
     "return t;"),
    ("paged_pool_rounds_up",
     "int64_t pool_blocks = (int64_t)ratio * R * D / hb;",
     "int64_t pool_blocks = ((int64_t)ratio * R * D + hb - 1) / hb;"),
    ("paged_missing_row_not_reported",
     "            *status = HSO_NO_HOST_ROW;\n            for (int j = 0; j < k; ++j) out[j] = -1;\n            free(done); free(is_hit_slot); free(miss);\n            return;",
     "            break;"),
    ("paged_backup_without_block",
     "        if (host_row_of(o, r, p) < 0) {\n            status[r] = HSO_NO_HOST_ROW;\n"
     "            note_status(o, r, status[r]);\n            continue;\n        }\n",
     ""),
    ("prefill_without_rows",
     "                if (host_row_of(o, r, S - n + i) < 0) { st = HSO_NO_HOST_ROW; break; }",
     "                ;"),
    ("protect_one_call_short",
     "uint32_t thr = tick > p ? tick - p : 1u;",
     "uint32_t thr = tick > p ? tick - p + 1u : 1u;"),
    ("protect_includes_prefill_stamps",
     "uint32_t thr = tick > p ? tick - p : 1u;",
     "uint32_t thr = tick > p ? tick - p : 0u;"),
    ("capacity_keeps_outputs",
     "            *status = HSO_CAPACITY;\n            for (int j = 0; j < k; ++j) out[j] = -1;",
     "            *status = HSO_CAPACITY;"),
    ("status_word_overwritten",
     "if (code != HSO_OK) o->status_word[r] |= (int32_t)1 << code;",
     "if (code != HSO_OK) o->status_word[r] = (int32_t)1 << code;"),
    ("status_word_cleared_by_success",
     "if (code != HSO_OK) o->status_word[r] |= (int32_t)1 << code;",
     "o->status_word[r] = code != HSO_OK ? (o->status_word[r] | ((int32_t)1 << code)) : 0;"),
    ("status_word_holds_code_not_bit",
     "if (code != HSO_OK) o->status_word[r] |= (int32_t)1 << code;",
     "if (code != HSO_OK) o->status_word[r] |= code;"),
    ("backup_error_not_recorded",
     "            status[r] = HSO_BAD_POSITION;\n            note_status(o, r, status[r]);",
     "            status[r] = HSO_BAD_POSITION;"),
    ("prefill_error_not_recorded",
     "        note_status(o, r, st);\n",
     ""),
    ("prefill_resets_other_requests",
     "        if (S == -1) continue;",
     "        if (S == -1) S = 0;"),
]


def run_all_pins(lib_path):
    """Names of the pins that reject the oracle at lib_path."""
    failed = []
    for n in names():
        try:
            if T.run_trace_on_oracle(n, lib_path) is not None:
                failed.append("golden:" + n)
        except Exception:
            failed.append("golden:" + n)
    for D, S, k, nc in [(3, 5, 2, 3), (4, 7, 3, 2)]:
        progs = T._exhaustive_programs(S, k, nc)
        try:
            if T.compare_with_model(D, k, [S] * len(progs), progs, lib_path) is not None:
                failed.append(f"exhaustive:{D},{S},{k}")
        except Exception:
            failed.append(f"exhaustive:{D},{S},{k}")
    for pin in T.PINS:
        try:
            pin(lib_path)
        except Exception:
            failed.append(pin.__name__)
    for seed in range(3):
        try:
            T.test_random_resident_tables_vs_list_model(seed, lib_path)
        except Exception:
            failed.append(f"resident_random:{seed}")
    for pin in TP.PAGED_PINS:
        try:
            pin(lib_path)
        except Exception:
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("mid,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, mid, orig, planted):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {mid} not unique"
    mut = tmp_path / f"oracle_{mid}.c"
    mut.write_text(src.replace(orig, planted))
    lib = tmp_path / f"liboracle_{mid}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-w", "-shared", "-fPIC",
                           "-o", str(lib), str(mut)])
    # run the pins in a child process: a planted mistake may also crash it
    here = os.path.dirname(os.path.abspath(__file__))
    code = ("import sys; sys.path[:0] = [%r, %r]; import test_oracle_mutants as M; "
            "f = M.run_all_pins(%r); print(f); sys.exit(3 if f else 0)"
            % (here, os.path.dirname(here), str(lib)))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode != 0, f"no pin rejects the planted mistake {mid}"


def test_unmodified_oracle_passes_all_pins():
    assert run_all_pins(O.build()) == []
