"""The bench's roofline accounting on the decode workload (32 sequences x
ctx 32,768, one query each at t = 32,767, K = 512 pools), against closed forms
written from the shapes: pooled keys 256 B per pool, 1024 B per attended latent
row (512 bf16 nope columns), q_idx 32 x 128 bf16 and w 32 fp32 per query,
q_lat and out 64 x 512 bf16 and lse 64 fp32 per query."""
import os
import sys

import kpool_inputs as KI

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

B, CTX, K = 32, 32768, 512


def test_decode_step_bytes_closed_form():
    wl = KI.make(KI.named("decode"))
    alg, n_tok = bench.algorithmic_bytes(wl)
    pools = CTX // 4                                   # t + 1 = 32,768: every pool full, no tail
    assert n_tok == B * K * 4
    assert alg["indexer_score"] == B * pools * 256 + B * (32 * 128 * 2 + 32 * 4)
    assert alg["sparse_mla_attend"] == B * K * 4 * 1024 + B * 64 * (512 * 2 + 512 * 2 + 4)
    assert alg["sparse_mla_attend"] == 71_311_360
    # one new token per sequence (key and gate rows) completes one pool
    assert alg["kpool_compress"] == B * (2 * 128 * 2) + B * 128 * 2
    assert alg["topk_select"] == 0                     # the score matrix is an intermediate of the step


def test_kernel_bytes_count_the_score_rows_top_k_reads():
    wl = KI.make(KI.named("decode"))
    alg, _ = bench.algorithmic_bytes(wl)
    kb = bench.kernel_bytes(wl, alg)
    assert kb["topk_select"] == B * (CTX // 4) * 4 + B * (K + 1) * 4
    assert kb["indexer_score_select"] == alg["indexer_score"] + B * (K + 1) * 4
    for st in ("kpool_compress", "indexer_score", "sparse_mla_attend"):
        assert kb[st] == alg[st]


def test_flops_closed_form():
    wl = KI.make(KI.named("decode"))
    fl = bench.algorithmic_flops(wl)
    assert fl["indexer_score"] == B * (CTX // 4) * 32 * 128 * 2
    assert fl["sparse_mla_attend"] == B * K * 4 * 64 * 512 * 2 * 2


def test_source_hash_follows_code_not_comments():
    a = "int f(int x) {  // doubles x\n    return 2 * x; /* fast */\n}\n"
    b = "// header comment\nint f(int x) {\n  return 2 * x;\n}\n"
    c = "int f(int x) { return 3 * x; }\n"
    assert bench.code_of(a) == bench.code_of(b)
    assert bench.code_of(a) != bench.code_of(c)
    for stage in bench.KERNEL_FILES:
        assert len(bench.kernel_source_hash(stage)) == 16
