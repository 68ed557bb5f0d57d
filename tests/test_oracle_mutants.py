"""Plausible mistakes planted in a copy of the oracle must fail a pin.

Each mutant is the oracle source with one textual change, compiled on the CPU
into a temporary library.  The pins are run against it; the test passes only
if at least one pin rejects the mutant.  The committed oracle is never
modified.
"""
import os
import tempfile

import pytest

import pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "hs_oracle.cpp")

MUTANTS = {
    "mru_victims": ("if (rc.ep[a] != rc.ep[b]) return rc.ep[a] < rc.ep[b];",
                    "if (rc.ep[a] != rc.ep[b]) return rc.ep[a] > rc.ep[b];"),
    "highest_slot_tie_break": ("if (rc.ep[a] != rc.ep[b]) return rc.ep[a] < rc.ep[b];\n        return a < b;",
                               "if (rc.ep[a] != rc.ep[b]) return rc.ep[a] < rc.ep[b];\n        return a > b;"),
    "hits_not_marked": ("for (int32_t v : hit_slots) rc.ep[v] = E;", ""),
    "oldest_step_preferred": ("return last_step[a] > last_step[b];",
                              "return last_step[a] < last_step[b];"),
    "last_step_not_updated": ("last_step[j] = s;\n                locs_b[i]",
                              "locs_b[i]"),
    "duplicate_at_wrong_row": ("locs_b[i] = (int32_t)(base + rc.phys[H + j]);",
                               "locs_b[i] = (int32_t)(base + rc.phys[j]);"),
    "off_by_one_validity": ("if (t < 0 || t >= limit)", "if (t < 0 || t > limit)"),
    "copy_without_rotation": ("std::swap(rc.phys[v], rc.phys[H + j]);", ""),
    "epoch_not_advanced": ("rc.epoch = E + 1;", "rc.epoch = E;"),
    "cap_ignores_hits": ("const int32_t cap = H - (int32_t)hit_slots.size();",
                         "const int32_t cap = H;"),
    "victims_paired_unsorted": ("cand.resize(m);\n    std::sort(cand.begin(), cand.end());",
                                "cand.resize(m);"),
    "row_from_request_zero": ("const int64_t src_row = (int64_t)q * o.L + t;",
                              "const int64_t src_row = t;"),
    "seq_len_ignored": ("const int32_t limit = std::min(seq_len, o.L);",
                        "const int32_t limit = o.L;"),
    "evictions_not_counted": ("stat[HSO_STAT_EVICTED]++;", ""),
    "extra_page_ignored": ("if (o.E > 0 && t >= extra_page_start(limit, o.E)) {",
                           "if (false) {"),
    "extra_page_starts_at_length": ("return (n - 1) / E * E;", "return n / E * E;"),
    "extra_row_ignores_request": ("(int64_t)q * o.E + t % o.E;", "t % o.E;"),
    "append_skips_extra_row": ("std::memcpy(device_kv + extra_row(*o, q, t) * W, row, (size_t)W);",
                               ";"),
    "append_skips_hot_copy": ("if (r != rc.res.end())\n            std::memcpy(",
                              "if (false)\n            std::memcpy("),
    "append_ignores_page": ("if (o->E > 0 && t >= extra_page_start(limit, o->E))",
                            "if (o->E > 0)"),
    "append_skips_host": ("std::memcpy(host_pool + ((int64_t)q * o->L + t) * W, row, (size_t)W);",
                          ";"),
    "hit_location_ignores_rotation": ("locs_b[i] = (int32_t)(base + rc.phys[v]);",
                                      "locs_b[i] = (int32_t)(base + v);"),
    "page_offset_dropped": ("? index[t / page_size] * page_size + t % page_size",
                            "? index[t / page_size] * page_size"),
    "invalid_not_counted": ("stat[HSO_STAT_INVALID]++;", ""),
    "overflow_tie_prefers_later_miss": ("return last_step[a] > last_step[b];\n            return a < b;",
                                        "return last_step[a] > last_step[b];\n            return a > b;"),
    "duplicate_misses_not_merged": ("auto f = first.find(t);", "auto f = first.end();"),
    "plan_source_is_destination": ("if (src_b) src_b[j] = src_row;", "if (src_b) src_b[j] = dst_row;"),
    "plan_count_off_by_one": ("if (count_b) *count_b = (int32_t)U.size();",
                              "if (count_b) *count_b = (int32_t)U.size() - 1;"),
    "layers_share_one_cache": ("swap_in_request(*o, o->at(layer, q), q,",
                               "swap_in_request(*o, o->at(0, q), q,"),
    "reset_first_layer_only": (
        "for (int32_t l = 0; l < o->layers; ++l) make_empty(*o, o->at(l, req_pool_indices[i]));",
        "make_empty(*o, o->at(0, req_pool_indices[i]));"),
    "reset_skips_first_request": (
        "    for (int32_t i = 0; i < n; ++i)\n        for (int32_t l = 0; l < o->layers; ++l)",
        "    for (int32_t i = 1; i < n; ++i)\n        for (int32_t l = 0; l < o->layers; ++l)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    from oracle.oracle import build_oracle, load_library
    old, new = MUTANTS[name]
    with open(ORACLE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, "mutation anchor not found once: %r" % old
    mutated = src.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "hs_oracle_mutant.cpp")
        with open(path, "w") as f:
            f.write(mutated)
        lib_path = build_oracle(src=path, out_path=os.path.join(d, "libmutant.so"), force=True)
        lib = load_library(lib_path)
        caught = []
        for pin in pins.ALL_PINS:
            try:
                pin(lib)
            except AssertionError as e:
                caught.append((pin.__name__, str(e)[:80]))
                break
        assert caught, "mutant %s passed every pin" % name
