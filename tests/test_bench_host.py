"""The benchmark's host-side accounting, checked without a GPU.

The algorithmic bytes are the roofline's numerator, so they are pinned to figures worked out by
hand from the block formats (a Q4_1 block is 20 bytes per 32 values, a Q4_K super-block 144
bytes per 256 values, a Q6_K one 210).
"""

import bench
from expert_ffn_decode_gb300 import synth


def test_flint_decode_bytes():
    w = synth.WORKLOADS["flint_decode_t1"]
    expert = 3 * 512 * (2048 // 32) * 20        # gate, up, down of one expert: 1,966,080
    shared = 3 * 1024 * (2048 // 32) * 20       # 3,932,160
    router = 256 * 2048 * 4                     # f32 router rows
    xo = 2 * 2048 * 4                           # x in, out
    assert bench.record_bytes(w, 512) == expert == 1966080
    assert bench.active_bytes(w) == 6 * expert + shared == 15728640
    assert bench.layer_bytes(w) == 6 * expert + shared + router + xo == 17842176


def test_kquant_record_bytes():
    w = synth.WORKLOADS["ling_kq_decode_t1"]
    gu = 2 * 768 * (2560 // 256) * 144          # Q4_K gate and up rows
    dn = 2560 * (768 // 256) * 210              # Q6_K down rows
    assert bench.record_bytes(w, 768) == gu + dn == 3824640
    assert bench.qtype_label(w) == "Q4_K/Q6_K"
    assert bench.qtype_label(synth.WORKLOADS["flint_decode_t1"]) == "Q4_1"


def test_batched_launch_count():
    # the tile path (all Q4_1 or all Q4_0 with K dimensions in whole chunks; Q4_K gate/up with
    # Q4_K or Q6_K down in whole super-blocks) launches eight kernels a pass, the general path seven
    assert bench.prefill_launches(synth.WORKLOADS["flint_prefill_t512"]) == 8
    assert bench.prefill_launches(synth.WORKLOADS["ling_kq_prefill_t512"]) == 8
    wide_q6 = {**synth.WORKLOADS["ling_kq_prefill_t512"], "expert_ff": 1024}  # Q6_K rows past 768 values
    assert bench.prefill_launches(wide_q6) == 7
    assert bench.prefill_launches({**wide_q6, "qtype_down": synth.Q4_K}) == 8
    odd = {**synth.WORKLOADS["flint_prefill_t512"], "hidden": 96, "expert_ff": 96, "shared_ff": 0}
    assert bench.prefill_launches(odd) == 7
    q40 = {**synth.WORKLOADS["flint_prefill_t512"], "qtype": synth.Q4_0}  # Q4_0 chunks are 256 values
    assert bench.prefill_launches(q40) == 8
    q40_odd = {**q40, "expert_ff": 384}
    assert bench.prefill_launches(q40_odd) == 7


def test_capture_hash_ignores_comments_only():
    a = 'int f(int x) { return x + 1; }  // one\n/* two */\nconst char* s = "a // b";\n'
    b = '// header\nint f(int x) {\n  return x + 1;\n}\nconst char* s = "a // b";  /* tail */\n'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "a // b";\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert '"a // b"' in bench.code_only(a)  # a comment marker inside a literal is kept
