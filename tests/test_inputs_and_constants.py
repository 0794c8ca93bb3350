"""The synthetic workloads carry the shapes the pages print (tests/golden/page_constants.json)."""
import json
import os

import numpy as np

import kpool_inputs as KI

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "page_constants.json")))["facts"]


def test_workload_constants_match_the_pages():
    assert KI.KPOOL == FACTS["index_kpool"]["value"]
    assert KI.INDEX_HEADS == FACTS["index_n_heads"]["value"]
    assert KI.INDEX_DIM == FACTS["index_head_dim"]["value"]
    assert KI.MLA_HEADS == FACTS["num_attention_heads"]["value"]
    assert KI.NOPE_DIM == FACTS["kv_lora_rank"]["value"]
    assert KI.LATENT_DIM == FACTS["latent_width"]["value"]
    assert KI.LATENT_DIM - KI.NOPE_DIM == FACTS["rotary_columns"]["value"]
    assert abs(KI.Spec("x", [1], [1]).sm_scale - FACTS["qk_head_dim"]["value"] ** -0.5) < 1e-12
    for name in ("decode", "ragged", "prefill", "long"):
        assert KI.named(name).topk_tokens == FACTS["index_topk"]["value"]


def test_tiny_workload_layout():
    wl = KI.make(KI.named("tiny"))
    assert wl.lens.tolist() == [258]
    assert wl.q_pos.tolist() == [254, 255, 256, 257]
    assert wl.prev_len.tolist() == [254] and wl.new_off.tolist() == [0, 4]
    assert wl.k_pools == 16 and wl.max_pools == 64
    assert (wl.latent[:, 512:] == 0).all()
    assert (wl.q_lat[:, :, 512:] == 0).all()
    assert wl.keys.shape == (258, 128) and wl.q_lat.shape == (4, 64, 576)


def test_seeded_inputs_are_deterministic():
    a = KI.make(KI.named("tiny"))
    b = KI.make(KI.named("tiny"))
    assert np.array_equal(KI.bits(a.latent), KI.bits(b.latent))
    assert np.array_equal(a.w.numpy(), b.w.numpy())


def test_ragged_lengths_not_multiples_of_kpool():
    spec = KI.named("ragged")
    spec.ragged_lo, spec.ragged_hi = 300, 700        # same draw rule, small
    wl = KI.make(spec)
    assert (wl.lens % 4 != 0).all() and wl.B == 8
    assert ((wl.lens >= 300) & (wl.lens <= 700)).all()
    assert wl.q_pos.tolist()[:2] == [wl.lens[0] - 2, wl.lens[0] - 1]
