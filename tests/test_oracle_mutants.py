"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutant is a copy of ``oracle/oracle.c`` with one plausible slip (a wrong
comparison, a dropped term, a shifted index, a skipped step), compiled into a
temporary directory.  The test requires that the substitution applies, that the
mutant compiles, and that at least one pin of ``oracle_pins`` fails on it.
"""
import os
import sys

import numpy as np

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "close_on_exceed_not_reach": [("if (open_bytes[g] >= cap)", "if (open_bytes[g] > cap)")],
    "no_first_bucket_cap": [("closed_count[g] == 0) ? first_cap_bytes : cap_bytes",
                             "closed_count[g] == 0) ? cap_bytes : cap_bytes")],
    "first_cap_shared_by_dtypes": [("closed_count[g] == 0) ? first_cap_bytes", "nb == 0) ? first_cap_bytes")],
    "initial_list_not_reversed": [("(order == ORDER_FWD_THEN_REVERSE) ? nb - 1 - b : b", "b")],
    "forward_iteration": [("(order == ORDER_REVERSE) ? nparams - 1 - k : k", "k")],
    "megatron_issue_forward": [("(order == ORDER_MEGATRON) ? nb - 1 - b : b", "b")],
    "no_padding": [("((off + pad_multiple - 1) / pad_multiple) * pad_multiple", "off")],
    "no_scaling": [("local[r][e] = rank_buf[r][e] * inv_w", "local[r][e] = rank_buf[r][e]")],
    "received_value_dropped": [("local[r][i] = msg[from][i - b] + local[r][i]", "local[r][i] = local[r][i]")],
    "local_value_dropped": [("local[r][i] = msg[from][i - b] + local[r][i]", "local[r][i] = msg[from][i - b]")],
    "all_gather_one_step_short": [("for (int32_t s = 0; s < W - 1; s++) {\n            for (int32_t r = 0; r < W; r++) {\n                int32_t c = mod(r - s, W);",
                                   "for (int32_t s = 0; s < W - 2; s++) {\n            for (int32_t r = 0; r < W; r++) {\n                int32_t c = mod(r - s, W);")],
    "ring_owner_shifted": [("int32_t c = mod(r - s - 1, W);", "int32_t c = mod(r - s, W);"),
                           ("int32_t c = mod(from - s - 1, W);", "int32_t c = mod(from - s, W);"),
                           ("int32_t c = mod(r - s, W);\n                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);\n                for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];\n                bytes_sent[r] += (uint64_t)(e - b) * sizeof(float);\n            }\n            for (int32_t r = 0; r < W; r++) {\n                int32_t from = mod(r - 1, W);\n                int32_t c = mod(from - s, W);",
                            "int32_t c = mod(r - s + 1, W);\n                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);\n                for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];\n                bytes_sent[r] += (uint64_t)(e - b) * sizeof(float);\n            }\n            for (int32_t r = 0; r < W; r++) {\n                int32_t from = mod(r - 1, W);\n                int32_t c = mod(from - s + 1, W);"),
                           ("int64_t b = chunk_begin(n, W, r), e = chunk_end(n, W, r);",
                            "int64_t b = chunk_begin(n, W, (r + 1) % W), e = chunk_end(n, W, (r + 1) % W);")],
    "floor_chunk_split": [("int64_t len = (n + W - 1) / W;", "int64_t len = n / W > 0 ? n / W : 1;")],
    "pack_no_zero_fill": [("        if (!accumulate)\n            for (int64_t e = 0; e < bucket_numel; e++) out[e] = 0.0f;\n", "")],
    "accumulate_ignored": [("                if (accumulate)\n", "                if (0)\n")],
    "bf16_misdecoded": [("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;")],
    "f16_bias_wrong": [("u = sign | ((ex + 112) << 23) | (man << 13);", "u = sign | ((ex + 111) << 23) | (man << 13);")],
    "unpack_writes_unused": [("            if (global_used && !global_used[s]) continue;\n", "")],
    "unpack_ignores_shard": [("            lo = chunk_begin(bucket_numel, W, w);\n", "")],
    "wire_sum_not_rounded": [("                local[r][i] = oracle_round_wire(oracle_wire_value(msg[from][i - b], wire) +\n"
                              "                                                    oracle_wire_value(local[r][i], wire), wire);",
                              "                local[r][i] = oracle_round_wire(oracle_wire_value(msg[from][i - b], wire), wire) + 0 * "
                              "local[r][i];")],
    "wire_divide_skipped": [("local[r][e] = oracle_round_wire(oracle_wire_value(c, wire) / (double)W, wire);",
                             "local[r][e] = c;")],
    "wire_ties_away": [("double q = rint(ax / quantum);", "double q = floor(ax / quantum + 0.5);")],
    "timeline_ignores_readiness": [("start_ms[b] = ready > comm_free ? ready : comm_free;", "start_ms[b] = comm_free;")],
    "timeline_serial_without_backward": [("*serial_ms = backward_end + comm_total;", "*serial_ms = comm_total;")],
    "rebuild_ignores_sequence": [("seq[k] = given ? given[k] :", "seq[k] = 0 ? given[k] :")],
    "bitmap_or_as_and": [("global_used[p] = sum > 0 ? 1 : 0;", "global_used[p] = sum == W ? 1 : 0;")],
    "bitmap_skips_last_replica": [("for (int32_t w = 0; w < W; w++) {\n            int32_t bit",
                                   "for (int32_t w = 0; w < W - 1; w++) {\n            int32_t bit")],
    "bitmap_counts_raw_bytes": [("int32_t bit = local_used[(int64_t)w * nparams + p] != 0 ? 1 : 0;",
                                 "int32_t bit = local_used[(int64_t)w * nparams + p];")],
    "bitmap_transposed_index": [("local_used[(int64_t)w * nparams + p] != 0", "local_used[(int64_t)p * W + w] != 0")],
    "offset_skips_first": [("            offset_of[p] = off;\n            off += numels[p];",
                            "            off += numels[p];\n            offset_of[p] = off - numels[p] + (j > 0);")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) >= 1, f"substitution for {name} no longer applies: {old!r}"
        src = src.replace(old, new, 1)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src)
    lib = oracle.build(str(path), str(tmp_path / "liboracle_mutant.so"), extra=("-w",))
    orc = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"


# ---------------------------------------------------------------------------
# the PowerSGD oracle (Python): each mutant is a patched copy of the module
# ---------------------------------------------------------------------------
PSGD_MUTANTS = {
    "p_not_all_reduced": [("p = sum(mw[w] @ q for w in range(W))\n", "p = mw[0] @ q\n")],
    "p_not_orthogonalised": [("        p = _orthonormal(p)\n", "")],
    "q_not_divided_by_world": [("qn = sum(mw[w].T @ p for w in range(W)) / W", "qn = sum(mw[w].T @ p for w in range(W))")],
    "error_not_fed_back": [("mw.append(g + state.error[w][t] if state.error_feedback else g)", "mw.append(g)")],
    "error_sign_flipped": [("state.error[w][t] = mw[w] - approx", "state.error[w][t] = approx - mw[w]")],
    "warm_start_dropped": [("        state.q[t] = qn\n", "")],
    "rank_not_clamped": [("    return min(rank, m, n)", "    return rank")],
    "vectors_left_alone": [("                out[:, seg_offset[t]:seg_offset[t] + k] = mean[:, pos:pos + k]", "                pass")],
    "warmup_ignored": [("    if state.iter < state.start_iter:", "    if False:")],
    "view_last_dim": [("    return shape[0], n", "    return n, shape[0]")],
    "qr_sign_not_fixed": [("    qm = qm * np.where(d < 0, -1.0, 1.0)\n", "")],
}


@pytest.mark.parametrize("name", sorted(PSGD_MUTANTS))
def test_powersgd_mutant_is_caught(name, tmp_path, orc):
    import importlib.util

    from oracle import powersgd
    from oracle_pins_powersgd import POWERSGD_PINS

    src = open(powersgd.__file__).read()
    for old, new in PSGD_MUTANTS[name]:
        assert src.count(old) >= 1, f"substitution for {name} no longer applies: {old!r}"
        src = src.replace(old, new, 1)
    path = tmp_path / f"powersgd_{name}.py"
    path.write_text(src)
    spec = importlib.util.spec_from_file_location(f"powersgd_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod          # dataclasses look the module up while it loads
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules[spec.name]
    failed = []
    for pin in POWERSGD_PINS:
        try:
            pin(orc, mod)
        except (AssertionError, ValueError, np.linalg.LinAlgError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
