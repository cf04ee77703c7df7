"""The oracle's pins catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake by text
substitution, compiles the copy on the CPU and checks that the hand-worked
example or the linked-list simulator comparison rejects it.  Nothing here
touches the real oracle or any GPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

# Dropping the explicit "skip slots hit this step" from the victim candidates
# is an equivalent change under LRU (hit slots already carry this step's
# stamp, the newest, and K <= S leaves enough older slots), but not under FIFO,
# where a hit keeps its old fill stamp: "fifo_hit_slots_evictable" plants it.

SRC = os.path.join(os.path.dirname(oracle.__file__), "hs_oracle.c")

MUTANTS = {
    "tie_break_highest_slot": ("if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;",
                               "if (x->slot != y->slot) return x->slot < y->slot ? 1 : -1;"),
    "hits_do_not_refresh": ("if (hit[s]) stamp[s] = step;", "if (0) stamp[s] = step;"),
    "victims_in_lru_order": ("qsort(victims, (size_t)nmiss, sizeof(int32_t), or_cmp_int);", ""),
    "victims_descending": ("int32_t v = victims[i];", "int32_t v = victims[nmiss - 1 - i];"),
    "evicted_token_kept": ("if (old >= 0) tok_slot[old] = -1;", "(void)old;"),
    "fill_not_stamped": ("        stamp[v] = step;\n", "\n"),
    "wrong_row_copied": ("host + (size_t)t * (size_t)R", "host + (size_t)v * (size_t)R"),
    "duplicates_accepted": ("if (seen[t]) {                               /* repeat", "if (0) {  /* repeat"),
    "duplicates_not_flagged": ("            else err |= OR_E_DUP;\n", "\n"),
    "range_off_by_one": ("t >= len || t >= C", "t > len || t >= C"),
    "tail_offset_from_start": ("out[j] = S + t % T;", "out[j] = S + (t - cold);"),
    "tail_counted_as_miss": ("            inplace += 1;\n", "\n"),
    "stamp_plus_one": ("if (hit[s]) stamp[s] = step;", "if (hit[s]) stamp[s] = step + 1;"),
    "fifo_refreshes_hits": ("if (policy != OR_POLICY_FIFO)\n", "if (1)\n"),
    "sliding_no_write_back": ("if (t >= T) memcpy(host", "if (0) memcpy(host"),
    "sliding_fixed_boundary": ("sliding ? (len - T > 0 ? len - T : 0) : C - T", "C - T"),
    "alias_repeats_unresolved": ("out[j] = out[alias_of[j]];", "out[j] = -1;"),
    "fifo_hit_slots_evictable": ("if (hit[s]) continue;", "if (0) continue;"),
    "evict_newest_first": ("if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;",
                           "if (x->stamp != y->stamp) return x->stamp > y->stamp ? -1 : 1;"),
    "misses_paired_reversed": [("int32_t t = miss_tok[i];", "int32_t t = miss_tok[nmiss - 1 - i];"),
                               ("out[miss_pos[i]] = v;", "out[miss_pos[nmiss - 1 - i]] = v;")],
    "short_row_copy": ("(size_t)t * (size_t)R, (size_t)R);", "(size_t)t * (size_t)R, (size_t)R - 1);"),
    "tail_boundary_off_by_one": ("if (t >= cold) {", "if (t > cold) {"),
    "padding_flagged": ("if (t == -1) continue;", "if (t == -1) { err |= OR_E_RANGE; continue; }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(tmp_path, name):
    edits = MUTANTS[name]
    if isinstance(edits, tuple):
        edits = [edits]
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src)
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", str(path), "-o", str(so)],
                   check=True)
    # Run the pins in a child process: a planted mistake may also crash.
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import oracle\n"
        "from test_oracle import check_golden, check_against_simulator\n"
        "lib = oracle.load_library(%r)\n"
        "try:\n"
        "    check_golden(oracle, lib=lib)\n"
        "    check_against_simulator(oracle, range(400), lib=lib)\n"
        "    check_against_simulator(oracle, range(150), lib=lib, fifo=True)\n"
        "    check_against_simulator(oracle, range(150), lib=lib, sliding=True)\n"
        "    check_against_simulator(oracle, range(150), lib=lib, alias=True)\n"
        "except AssertionError:\n"
        "    sys.exit(3)\n"
        "sys.exit(0)\n" % (here, os.path.dirname(here), str(so)))
    rc = subprocess.run([sys.executable, "-c", code], capture_output=True).returncode
    assert rc != 0, "planted mistake %s passed every pin" % name


# Random eviction: each planted mistake must fail the random-policy pins
# (tests/test_oracle_random.py: the generator's published outputs, the
# invariants, the uniform spread, the dependence on request and seed).
RANDOM_MUTANTS = {
    "random_key_ignores_request": ("((uint64_t)(uint32_t)req << 14)", "((uint64_t)0 << 14)"),
    "random_key_ignores_seed": ("or_splitmix64(seed ^ x)", "or_splitmix64(x)"),
    "random_empty_not_first": ("    if (empty) return 0;\n", "\n"),
    "random_generator_constant": ("z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;",
                                  "z = (z ^ (z >> 27)) * 0x94D049BB133111EAull;"),
    "random_hits_not_refreshed": ("if (policy != OR_POLICY_FIFO)\n", "if (policy == OR_POLICY_LRU)\n"),
    "random_keys_by_slot": ("return 1 + (int32_t)(or_splitmix64(seed ^ x) >> 34);", "return 1 + s;"),
}


@pytest.mark.parametrize("name", sorted(RANDOM_MUTANTS))
def test_random_pins_reject_planted_mistake(tmp_path, name):
    old, new = RANDOM_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    src = src.replace(old, new)
    path = tmp_path / ("mut_%s.c" % name)
    path.write_text(src)
    so = tmp_path / ("libmut_%s.so" % name)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-w", str(path), "-o", str(so)],
                   check=True)
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import oracle\n"
        "from test_oracle_random import check_random\n"
        "lib = oracle.load_library(%r)\n"
        "try:\n"
        "    check_random(lib)\n"
        "except AssertionError:\n"
        "    sys.exit(3)\n"
        "sys.exit(0)\n" % (here, os.path.dirname(here), str(so)))
    rc = subprocess.run([sys.executable, "-c", code], capture_output=True).returncode
    assert rc != 0, "planted mistake %s passed every random-policy pin" % name
