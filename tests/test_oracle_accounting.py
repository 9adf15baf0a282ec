"""Pins of the oracle's byte/bit accounting against the numbers the pages print."""
import json
import os

import pytest

from oracle import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "accounting.json")))


def test_kivi_worked_example_bytes_per_token():
    e = GOLD["kivi_llama2_7b"]
    b = acc.kv_cache_bytes(e["n_layer"], e["h_kv"], e["d_head"], 1, e["bytes_per_elem"])
    assert b == e["bytes_per_token"] == 524288


def test_kivi_worked_example_context_and_batch():
    e = GOLD["kivi_llama2_7b"]
    ctx = acc.kv_cache_bytes(e["n_layer"], e["h_kv"], e["d_head"], e["context"], e["bytes_per_elem"])
    assert ctx == e["bytes_per_context"] == 2 * 2**30            # "2 GB" per 4K context
    assert ctx * e["batch"] == e["bytes_per_batch"] == 32 * 2**30  # "32 GB" at batch 16


@pytest.mark.parametrize("row", GOLD["loopvq"])
def test_vq_bits_per_element(row):
    assert acc.vq_bits_per_element(row["code_bits"], row["G"]) == row["bits_per_elem"]


@pytest.mark.parametrize("T,Tc,G,D,bits", [(4, 2, 16, 128, 0.5), (4, 4, 32, 128, 0.25),
                                           (4, 1, 16, 128, 0.5), (32, 4, 16, 128, 0.5)])
def test_loopvq_index_bytes_match_bits(T, Tc, G, D, bits):
    # loop-axis coupling keeps the bitwidth at b/G (LoopVQ method, core innovations)
    per_tok = acc.loopvq_index_bytes_per_token_head(T, Tc, G, D)
    assert per_tok * 8 / (T * D) == bits


def test_kivi_bits_and_ratio():
    e = GOLD["kivi_2bit"]
    bpe = acc.kivi_bits_per_element(e["bits"], e["group"])
    assert bpe == e["bits_per_elem"]
    assert bpe / 8 == e["bytes_per_elem"]
    assert round(16 / bpe, 1) == e["fp16_ratio_approx"]
