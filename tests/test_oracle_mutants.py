"""Plant one plausible mistake at a time in a copy of the oracle's C source,
build it, and require that the pins catch it.  This shows the pins are tight
enough that a dropped term, a wrong index, a reversed comparison or a
transposed operand anywhere in the oracle would not go unnoticed.

Each mutant runs in its own process: a mistake that reads out of bounds must
not take the test run down with it (a crash counts as caught)."""
import os
import subprocess
import sys
import tempfile

import pytest

from oracle import build as obuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in the oracle, replacement)
MUTANTS = [
    ("sort_descending",
     "num_sched[order[k]] > num_sched[cur]", "num_sched[order[k]] < num_sched[cur]"),
    ("ties_reversed",
     "num_sched[order[k]] > num_sched[cur]", "num_sched[order[k]] >= num_sched[cur]"),
    ("no_sort",
     "index_mapping[b] = rows[order[b]];\n        nb[b] = num_sched[order[b]];",
     "index_mapping[b] = rows[b];\n        nb[b] = num_sched[b];"),
    ("mapping_unsorted",
     "index_mapping[b] = rows[order[b]];", "index_mapping[b] = rows[b];"),
    ("qsl_unsorted_counts",
     "query_start_loc[b + 1] = query_start_loc[b] + nb[b];",
     "query_start_loc[b + 1] = query_start_loc[b] + num_sched[b];"),
    ("seq_lens_drop_new",
     "seq_lens[b] = st->completed[index_mapping[b]] + nb[b];",
     "seq_lens[b] = st->completed[index_mapping[b]];"),
    ("position_from_zero",
     "int32_t p = st->completed[r] + k;", "int32_t p = k;"),
    ("ids_chunk_relative",
     "input_ids[t] = st->tok[r][p];", "input_ids[t] = st->tok[r][k];"),
    ("slot_drop_offset",
     "(int64_t)physical * bsz + offset;", "(int64_t)physical * bsz;"),
    ("slot_logic_block",
     "(int64_t)physical * bsz + offset;", "(int64_t)logic_block * bsz + offset;"),
    ("slot_times_width",
     "(int64_t)physical * bsz + offset;", "(int64_t)physical * st->W[g] + offset;"),
    ("offset_swapped",
     "int32_t offset = p % bsz;", "int32_t offset = p / bsz;"),
    ("lookup_wrong_row",
     "int32_t physical = st->bt[g][(int64_t)r * st->W[g] + logic_block];",
     "int32_t physical = st->bt[g][(int64_t)b * st->W[g] + logic_block];"),
    ("tables_schedule_order",
     "st->bt[g][(int64_t)index_mapping[b] * st->W[g] + j];",
     "st->bt[g][(int64_t)rows[b] * st->W[g] + j];"),
    ("pages_floor",
     "int32_t pages = (int32_t)(((int64_t)seq_lens[b] + bsz - 1) / bsz);",
     "int32_t pages = (int32_t)((int64_t)seq_lens[b] / bsz);"),
    ("last_page_remainder",
     "last_page_len[b] = seq_lens[b] - (pages - 1) * bsz;",
     "last_page_len[b] = seq_lens[b] % bsz;"),
    ("indptr_counts_width",
     "kv_indptr[b + 1] = kv_indptr[b] + pages;", "kv_indptr[b + 1] = kv_indptr[b] + st->W[g];"),
    ("indices_batch_row",
     "kv_indices[kv_indptr[b] + j] = st->bt[g][(int64_t)r * st->W[g] + j];",
     "kv_indices[kv_indptr[b] + j] = st->bt[g][(int64_t)b * st->W[g] + j];"),
    ("capacity_off_by_one",
     "if (total > capacity || total > INT32_MAX) return OR_BAD_ARG;",
     "if (total >= capacity || total > INT32_MAX) return OR_BAD_ARG;"),
    ("advance_by_one",
     "st->completed[index_mapping[b]] += nb[b];", "st->completed[index_mapping[b]] += 1;"),
    ("highest_free_row",
     "for (int32_t r = 0; r < st->rows; r++)\n        if (!st->active[r]) { row = r; break; }",
     "for (int32_t r = st->rows - 1; r >= 0; r--)\n        if (!st->active[r]) { row = r; break; }"),
    ("remove_keeps_table",
     "for (int32_t j = 0; j < st->W[g]; j++) line[j] = -1;\n        st->nblk",
     "for (int32_t j = 0; j < 0; j++) line[j] = -1;\n        st->nblk"),
    ("update_overwrites",
     "line[have + j] = new_block_ids[off + j];", "line[j] = new_block_ids[off + j];"),
    ("kv_v_from_k",
     "memcpy(v_cache + s * line_bytes, v + (int64_t)t * v_stride_bytes",
     "memcpy(v_cache + s * line_bytes, k + (int64_t)t * k_stride_bytes"),
    ("kv_ignores_stride",
     "k + (int64_t)t * k_stride_bytes, (size_t)line_bytes);",
     "k + (int64_t)t * line_bytes, (size_t)line_bytes);"),
    ("fnv_xor_after_multiply",
     "h ^= bytes[i];\n        h *= OR_FNV_PRIME;", "h *= OR_FNV_PRIME;\n        h ^= bytes[i];"),
    ("keys_not_chained",
     "prev = prev * OR_FNV_PRIME + digest;", "prev = digest;"),
    ("keys_big_endian",
     "buf[4 * k + 0] = (uint8_t)(t & 0xff);", "buf[4 * k + 0] = (uint8_t)((t >> 24) & 0xff);"),
    ("keys_partial_block",
     "int32_t nfull = n_tokens / block_size;", "int32_t nfull = (n_tokens + block_size - 1) / block_size;"),
    ("hits_no_cap",
     "int32_t cap = (n_tokens - 1) / block_size;", "int32_t cap = n_tokens / block_size;"),
    ("hits_skip_gaps",
     "if (found < 0) break;", "if (found < 0) continue;"),
    ("alloc_no_watermark",
     "if (new_blocks[g] + watermark > available) refused = 1;",
     "if (new_blocks[g] > available) refused = 1;"),
    ("alloc_pop_from_bottom",
     "line[have + k] = st->pool[g][st->pool_count[g]];",
     "line[have + k] = st->pool[g][k];"),
    ("alloc_no_lookahead",
     "return (int64_t)st->completed[r] + num_new + lookahead;",
     "return (int64_t)st->completed[r] + num_new;"),
    # the window frees of a request reach the stack only after its check
    # (a refused request still frees), or only after its allocation
    ("alloc_frees_after_check",
     [("        if (window) free_out_of_window(st, r, window);\n        /* (3)", "        /* (3)"),
      ("        if (refused) { admitted = i; break; }",
       "        if (window) free_out_of_window(st, r, window);\n"
       "        if (refused) { admitted = i; break; }")]),
    ("alloc_frees_after_allocation",
     [("        if (window) free_out_of_window(st, r, window);\n        /* (3)", "        /* (3)"),
      ("        if (refused) { admitted = i; break; }",
       "        if (refused) { if (window) free_out_of_window(st, r, window); admitted = i; break; }"),
      ("            if (out_new_blocks) out_new_blocks[i * st->G + g] = new_blocks[g];\n        }\n",
       "            if (out_new_blocks) out_new_blocks[i * st->G + g] = new_blocks[g];\n        }\n"
       "        if (window) free_out_of_window(st, r, window);\n")]),
    ("window_off_by_one",
     "int64_t start = (int64_t)st->completed[r] - (window[g] - 1);",
     "int64_t start = (int64_t)st->completed[r] - window[g];"),
    ("refused_keeps_going",
     "if (refused) { admitted = i; break; }",
     "if (refused) { continue; }"),
    ("alloc_duplicate_rows_accepted",
     "if (rows[k] == r) return OR_BAD_ARG;", "if (rows[k] == r) continue;"),
    ("release_skips_reset",
     "                if (line[j] >= 0) pool_push(st, g, line[j]);\n                line[j] = -1;",
     "                if (line[j] >= 0) pool_push(st, g, line[j]);"),
    ("kv_short_line",
     "memcpy(k_cache + s * line_bytes, k + (int64_t)t * k_stride_bytes, (size_t)line_bytes);",
     "memcpy(k_cache + s * line_bytes, k + (int64_t)t * k_stride_bytes, (size_t)line_bytes - 1);"),
]


@pytest.fixture(scope="module")
def mutant_results():
    src = open(obuild.SOURCE).read()
    tmp = tempfile.mkdtemp(prefix="pkv_mutants_")
    procs = {}
    for name, *edit in MUTANTS:
        # one (old, new) replacement, or a list of them applied in turn
        edits = edit[0] if len(edit) == 1 else [tuple(edit)]
        text = src
        for old, new in edits:
            assert text.count(old) >= 1, f"mutation site for {name} not found in the oracle"
            text = text.replace(old, new, 1)
        assert text != src
        c_path = os.path.join(tmp, f"{name}.c")
        so_path = os.path.join(tmp, f"lib_{name}.so")
        with open(c_path, "w") as f:
            f.write(text)
        obuild.build(c_path, so_path, force=True)
        procs[name] = subprocess.Popen(
            [sys.executable, os.path.join(ROOT, "tests", "oracle_pins.py"), so_path],
            cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    results = {}
    for name, p in procs.items():
        out, _ = p.communicate(timeout=300)
        results[name] = (p.returncode, out.decode(errors="replace"))
    return results


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant_results, name):
    rc, out = mutant_results[name]
    assert rc != 0, f"mutant {name} passed every pin:\n{out}"
