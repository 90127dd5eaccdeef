"""Plant plausible mistakes in the oracle (CPU only) and check the pins in
test_oracle.py catch every one of them.  A pin suite that lets a dropped
term, a wrong index or a transposed operand through would not be a pin."""
import math

import numpy as np
import pytest

import oracle
import oracle.smla_oracle as so
import tests.test_oracle as pins

PIN_CALLS = [
    pins.test_e4m3_table_matches_torch_all_codes,
    pins.test_e4m3_spec_values,
    pins.test_bf16_widen_matches_torch,
    pins.test_parse_rows_roundtrip_known_values,
    pins.test_index_worked_examples,
    lambda: pins.test_index_matches_append_simulation(2, 4, [13, 1, 9], 1),
    lambda: pins.test_index_matches_append_simulation(3, 2, [7, 2, 11], 1),
    lambda: pins.test_index_matches_append_simulation(4, 4, [77, 30], 3),
    pins.test_index_interleave_is_a_bijection_onto_rank_local_positions,
    lambda: pins.test_attention_dense_matches_torch_sdpa(7, 16),
    pins.test_attention_q_zero_closed_form,
    pins.test_attention_single_slot_closed_form,
    pins.test_merge_matches_torch_logsumexp,
    pins.test_merge_identity_changes_nothing_and_no_nan,
    pins.test_merge_all_empty_is_identity,
    pins.test_merge_of_shards_equals_unsharded_with_empty_shards,
    pins.test_topk_select_matches_torch_topk_on_distinct_scores,
    pins.test_topk_select_k1_is_numpy_argmax_with_ties,
    pins.test_topk_select_all_equal_scores_keep_the_first_positions,
    pins.test_topk_select_short_rows_keep_every_candidate,
    lambda: pins.test_dcp_topk_merge_of_rank_local_topk_equals_unsharded(4, 16, 1),
    lambda: pins.test_dense_decode_sharded_and_merged_matches_torch_causal_sdpa(2, 2, 1),
    pins.test_dense_decode_spec_tokens_equal_single_token_requests,
    pins.test_flatten_lse_matches_torch_permute_reshape,
]


def _e4m3_bias8(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -7
    return s * (1 + m / 8.0) * 2.0 ** (e - 8)


def _e4m3_no_subnormal(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    if e == 15 and m == 7:
        return math.nan
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def _parse_tiled_scales(rows):
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    scales = np.ascontiguousarray(rows[:, 512:528]).view("<f4").astype(np.float64)
    nope = so.e4m3_to_f64(rows[:, :512]) * np.tile(scales, 128)  # wrong index
    return nope, so.bf16_bits_to_f64(np.ascontiguousarray(rows[:, 528:]).view("<u2"))


def _parse_swapped_parts(rows):
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    scales = np.ascontiguousarray(rows[:, 640:656]).view("<f4").astype(np.float64)
    nope = so.e4m3_to_f64(rows[:, :512]) * np.repeat(scales, 128, axis=1)
    return nope, so.bf16_bits_to_f64(np.ascontiguousarray(rows[:, 512:640]).view("<u2"))


def _convert(variant):
    def f(req_id, block_table, topk, D, rank, block_size, interleave=1):
        topk = np.asarray(topk, dtype=np.int64)
        bt = np.asarray(block_table, dtype=np.int64)
        out = np.full(topk.shape, -1, dtype=np.int64)
        I = interleave
        for i in range(topk.shape[0]):
            t = topk[i]
            if variant == "interleave_owner_by_position":
                mine = (t >= 0) & (t % D == rank)
            else:
                mine = (t >= 0) & ((t // I) % D == rank)
            tm = t[mine]
            if variant == "no_div":
                lp = tm
            elif variant == "interleave_local_as_plain":
                lp = tm // D
            else:
                lp = (tm // (I * D)) * I + tm % I
            lp = np.minimum(lp, bt.shape[1] * block_size - 1)
            phys = bt[int(req_id[i]), lp // block_size]
            if variant == "no_mod":
                out[i, mine] = phys * block_size
            elif variant == "block_major":
                out[i, mine] = phys + (lp % block_size) * bt.max()
            else:
                out[i, mine] = phys * block_size + lp % block_size
            if variant == "keep_foreign":
                out[i, (t >= 0) & ~mine] = t[(t >= 0) & ~mine]
        return out.astype(np.int32), (out >= 0).sum(1).astype(np.int32)
    return f


def _topk_variant(variant):
    def f(scores, n_cand, K):
        scores = np.asarray(scores, dtype=np.float64)
        out = np.full((scores.shape[0], K), -1, dtype=np.int64)
        for i in range(scores.shape[0]):
            n = scores.shape[1] if variant == "no_bound" else int(n_cand[i])
            pos = np.arange(n)
            if variant == "ascending":
                order = np.lexsort((pos, scores[i, :n]))
            elif variant == "ties_last_first":
                order = np.lexsort((-pos, -scores[i, :n]))
            else:
                order = np.lexsort((pos, -scores[i, :n]))
            keep = order[:K]
            out[i, :len(keep)] = pos[keep]
        return out.astype(np.int32)
    return f


_MERGE = so.dcp_topk_merge  # the real merge, bound before any patching


def _topk_merge_first_rank(cand_ids, cand_scores, K):
    return _MERGE(cand_ids[:1], cand_scores[:1], K)


def _dense_variant(variant):
    def f(q_bits, pool, block_table, ctx, S, D, rank, block_size, sm_scale, interleave=1):
        ctx = np.asarray(ctx, dtype=np.int64)
        T, H = ctx.shape[0] * S, q_bits.shape[1]
        out, lse = np.zeros((T, H, 512)), np.full((T, H), -np.inf)
        for b in range(ctx.shape[0]):
            for s_ in range(S):
                i = b * S + s_
                if variant == "excludes_own":
                    p = int(ctx[b]) - S + s_ - 1
                else:  # "no_causal": every token sees the whole context
                    p = int(ctx[b]) - 1
                pos = np.arange(p + 1, dtype=np.int32)[None]
                slots, _ = so.dcp_filter_convert_index(np.array([b]), block_table, pos, D, rank,
                                                       block_size, interleave)
                mine = slots[0][slots[0] >= 0]
                out[i], lse[i] = so.sparse_mla_decode_rows(so.bf16_bits_to_f64(q_bits[i]),
                                                           np.asarray(pool)[mine], sm_scale)
        return out, lse
    return f


def _flatten_transposed(lse_bhs):
    lse_bhs = np.asarray(lse_bhs)
    B, H, S = lse_bhs.shape
    flat = np.empty((B * S, H), dtype=lse_bhs.dtype)
    for b in range(B):
        for s_ in range(S):
            flat[s_ * B + b] = lse_bhs[b, :, s_]
    return flat


def _rows_variant(variant):
    def f(q_row, rows, sm_scale):
        H = q_row.shape[0]
        if rows.shape[0] == 0:
            return np.zeros((H, 512)), np.full(H, -np.inf)
        nope, rope = so.parse_rows(rows)
        k = np.concatenate([nope, rope], axis=1)
        scale = 1.0 if variant == "no_scale" else sm_scale
        if variant == "rope_negated":
            k = np.concatenate([nope, -rope], axis=1)
        s = scale * (q_row @ k.T)
        m = s.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
        if variant == "log2":
            lse = lse / math.log(2.0)
        if variant == "no_max_in_lse":
            lse = np.log(np.exp(s - m).sum(axis=1))
        p = np.exp(s - lse[:, None])
        if variant == "softmax_over_heads":
            p = np.exp(s - np.log(np.exp(s).sum(axis=0, keepdims=True)))
        return p @ nope, lse
    return f


def _merge_variant(variant):
    def f(outs, lses):
        L = np.stack([np.asarray(x, dtype=np.float64) for x in lses])
        O = np.stack([np.asarray(x, dtype=np.float64) for x in outs])
        with np.errstate(all="ignore"):
            M = L.max(axis=0)
            w = np.exp(L - M[None])
            total = w.sum(axis=0)
            lse = M + np.log(total) if variant != "drop_max" else np.log(total)
            if variant == "unnormalised":
                weight = w
            else:
                weight = w / total[None]
            out = (weight[..., None] * O).sum(axis=0)
        return out, lse
    return f


MUTANTS = {
    "e4m3_bias8": ("E4M3_TABLE", np.array([_e4m3_bias8(c) for c in range(256)])),
    "e4m3_no_subnormal": ("E4M3_TABLE",
                          np.array([_e4m3_no_subnormal(c) for c in range(256)])),
    "parse_tiled_scales": ("parse_rows", _parse_tiled_scales),
    "parse_swapped_parts": ("parse_rows", _parse_swapped_parts),
    "convert_no_div": ("dcp_filter_convert_index", _convert("no_div")),
    "convert_no_mod": ("dcp_filter_convert_index", _convert("no_mod")),
    "convert_block_major": ("dcp_filter_convert_index", _convert("block_major")),
    "convert_keep_foreign": ("dcp_filter_convert_index", _convert("keep_foreign")),
    "convert_interleave_local_as_plain": ("dcp_filter_convert_index",
                                          _convert("interleave_local_as_plain")),
    "convert_interleave_owner_by_position": ("dcp_filter_convert_index",
                                             _convert("interleave_owner_by_position")),
    "topk_ascending": ("topk_select", _topk_variant("ascending")),
    "topk_ties_last_first": ("topk_select", _topk_variant("ties_last_first")),
    "topk_no_candidate_bound": ("topk_select", _topk_variant("no_bound")),
    "topk_merge_first_rank_only": ("dcp_topk_merge", _topk_merge_first_rank),
    "dense_excludes_own_position": ("dense_mla_decode", _dense_variant("excludes_own")),
    "dense_no_causal_mask": ("dense_mla_decode", _dense_variant("no_causal")),
    "flatten_transposed": ("flatten_lse_bhs", _flatten_transposed),
    "attn_no_scale": ("sparse_mla_decode_rows", _rows_variant("no_scale")),
    "attn_rope_negated": ("sparse_mla_decode_rows", _rows_variant("rope_negated")),
    "attn_log2": ("sparse_mla_decode_rows", _rows_variant("log2")),
    "attn_no_max_in_lse": ("sparse_mla_decode_rows", _rows_variant("no_max_in_lse")),
    "attn_softmax_over_heads": ("sparse_mla_decode_rows",
                                _rows_variant("softmax_over_heads")),
    "merge_drop_max": ("lse_merge", _merge_variant("drop_max")),
    "merge_unnormalised": ("lse_merge", _merge_variant("unnormalised")),
    "merge_nan_on_empty": ("lse_merge", _merge_variant("plain")),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(so, attr, repl)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, repl)
    if attr == "E4M3_TABLE":
        monkeypatch.setattr(so, "e4m3_to_f64",
                            lambda c: repl[np.asarray(c, dtype=np.uint8)])
        monkeypatch.setattr(oracle, "e4m3_to_f64",
                            lambda c: repl[np.asarray(c, dtype=np.uint8)])
    caught = []
    for call in PIN_CALLS:
        try:
            with np.errstate(all="ignore"):
                call()
        except (AssertionError, IndexError, ValueError):
            caught.append(call)
    assert caught, f"no pin caught mutant {name}"
