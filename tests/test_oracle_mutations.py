"""Plant plausible mistakes in the numpy oracle and check the pins catch each.

Each mutant is the oracle's own source with one edit (a wrong index, a dropped
term, a swapped operand), executed as a separate module on the CPU.  The pin
tests of ``test_oracle_pins`` are run against it; at least one must fail.
"""
import inspect
import types

import pytest

import test_oracle_pins as pins
from oracle import reference

MUTATIONS = {
    "gqa_head_modulo": ("return h // (num_heads // num_kv_heads)", "return h % num_kv_heads"),
    "gqa_head_times": ("return h // (num_heads // num_kv_heads)", "return min(h * (num_heads // num_kv_heads), num_kv_heads - 1)"),
    "logical_block_by_mod": ("logical = t // block_size", "logical = t % block_size"),
    "offset_shifted": ("return int(table_row[logical]), t % block_size", "return int(table_row[logical]), (t + 1) % block_size"),
    "offset_is_logical": ("return int(table_row[logical]), t % block_size", "return int(table_row[logical]), logical"),
    "ceil_as_floor": ("blocks = -(-tokens // block_size)", "blocks = tokens // block_size"),
    "unused_sign": ("return blocks, blocks * block_size - tokens", "return blocks, tokens - blocks * block_size"),
    "scale_dropped": ("x = scale * (K @ qd[s, h])", "x = (K @ qd[s, h])"),
    "scale_squared": ("x = scale * (K @ qd[s, h])", "x = scale * scale * (K @ qd[s, h])"),
    "key_value_swapped": ("x = scale * (K @ qd[s, h])", "x = scale * (V @ qd[s, h])"),
    "norm_dropped": ("out[s, h] = (w @ V) / w.sum()", "out[s, h] = (w @ V)"),
    "last_token_dropped": ("for t in range(L)]", "for t in range(L - 1)]"),
    "first_token_dropped": ("for t in range(L)]", "for t in range(1, L)]"),
    "max_not_subtracted_sign": ("w = np.exp(x - x.max())", "w = np.exp(x.max() - x)"),
    "slot_uses_offset_only": ("return pid * block_size + off", "return pid + off * block_size"),
    "write_transposed": ("pid, off = divmod(slot, B)", "off, pid = divmod(slot, B)"),
    "copy_reversed": ("k_cache[dst] = k_cache[src].clone()", "k_cache[src] = k_cache[dst].clone()"),
    "write_skips_zero_slot": ("if slot < 0:", "if slot <= 0:"),
    "prefill_not_causal": ("end = p + 1        # it sees tokens 0 .. p", "end = L"),
    "prefill_excludes_itself": ("end = p + 1        # it sees tokens 0 .. p", "end = p"),
    "prefill_position_from_start": ("p = L - n + i      # this query row's position", "p = i      # this query row's position"),
    "prefill_wrong_query_row": ("z = scale * (Kc @ qd[qs[s] + i, h])", "z = scale * (Kc @ qd[qs[s], h])"),
    "prefill_scale_dropped": ("z = scale * (Kc @ qd[qs[s] + i, h])", "z = (Kc @ qd[qs[s] + i, h])"),
}

PIN_TESTS = [
    (pins.test_block_layout_golden, {}),
    (pins.test_block_layout_tail_bound, {}),
    (pins.test_lookup_golden, {}),
    (pins.test_decode_identity_layout_matches_sdpa, {"Hq": 8, "Hkv": 2}),
    (pins.test_decode_invariant_under_block_relabelling, {"dtype": pins.torch.float32}),
    (pins.test_decode_shared_equals_private_copy, {}),
    (pins.test_decode_closed_forms, {}),
    (pins.test_decode_gqa_group_mapping, {}),
    (pins.test_write_kv_identity_slots, {"dtype": pins.torch.float16}),
    (pins.test_write_kv_skips_negative_and_rejects_outside, {}),
    (pins.test_copy_blocks, {}),
    (pins.test_prefill_identity_layout_matches_sdpa, {"Hq": 8, "Hkv": 2}),
    (pins.test_prefill_closed_forms, {}),
]


def _mutant(old: str, new: str) -> types.ModuleType:
    src = inspect.getsource(reference)
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _slot_pin(mod):
    assert list(mod.slot_mapping([[5, 1, 7]], [0], [9], 4)) == [29]


def test_unmutated_oracle_passes_every_pin():
    for fn, kw in PIN_TESTS:
        fn(reference, **kw)
    _slot_pin(reference)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name):
    mod = _mutant(*MUTATIONS[name])
    caught = []
    for fn, kw in PIN_TESTS + [(lambda m: _slot_pin(m), {})]:
        try:
            fn(mod, **kw)
        except Exception as e:  # noqa: BLE001 - any failure counts as detection
            caught.append(type(e).__name__)
    assert caught, f"no pin detects mutation {name}"
