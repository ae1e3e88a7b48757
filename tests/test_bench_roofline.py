"""The bench's roofline arithmetic, recounted by hand from the 1.7B
predictor's shapes: the algorithmic bytes and FLOPs one call moves and
computes, and the engine the automatic choice names for each configuration.
"""
import bench
import synthetic as S


def _hand_count():
    # per layer: q|k|v rows 16*128 + 2*8*128 over hidden 1024, O 1024 x 2048,
    # gate and up 2 x 3072 x 1024, down 1024 x 3072
    layer = (2048 + 2048) * 1024 + 1024 * 2048 + 2 * 3072 * 1024 + 1024 * 3072
    head, proj = 2048 * 1024, 1024 * 2048
    matrices = 15 * (5 * layer + head) + proj
    frame_io = 2048 * 4 + 4 + 15 * 4 + 2048 * 2 + 14 * 1024 * 2
    return layer, matrices, frame_io


def test_algorithmic_bytes_match_a_hand_count():
    g = S.Geometry()
    layer, matrices, frame_io = _hand_count()
    assert layer == 15_728_640 and frame_io == 41_024
    for B in (1, 32, 128):
        nbytes, _ = bench.work_of(g, B, "bf16", sampling=False)
        assert nbytes == 2 * matrices + B * frame_io
    assert bench.work_of(g, 1, "bf16", False)[0] == 2_426_445_888
    assert bench.work_of(g, 32, "bf16", False)[0] == 2_427_717_632
    # Q8_0: 32 int8 weights and one f16 scale per block
    assert bench.work_of(g, 1024, "q8_0", False)[0] == matrices * 34 / 32 + 1024 * frame_io
    # sampling adds the Gumbel noise: one f32 per logit, step and frame
    assert bench.work_of(g, 256, "bf16", True)[0] == 2 * matrices + 256 * (frame_io + 15 * 2048 * 4)


def test_flops_count_every_position_and_the_attention():
    g = S.Geometry()
    layer, _, _ = _hand_count()
    attn = sum(5 * 16 * (p + 1) * 128 * 4 for p in range(16))   # q.k and p.v over p + 1 keys, 16 q heads
    per_frame = 2 * 16 * 5 * layer + 2 * 15 * 2048 * 1024 + 2 * 2 * 1024 * 2048 + attn
    for B in (1, 256):
        assert bench.work_of(g, B, "bf16", False)[1] == B * per_frame


def test_roofline_picks_the_binding_roof():
    g = S.Geometry()
    hbm, tf = 6696.8, 1907.6
    small = bench.roofline_of(g, 1, "bf16", False, 1.0, hbm, tf)
    assert small["bound"] == "hbm" and small["unit"] == "GB/s"
    assert abs(small["achieved"] - bench.work_of(g, 1, "bf16", False)[0] / 1e-3 / 1e9) < 1e-6
    big = bench.roofline_of(g, 1024, "q8_0", False, 10.0, hbm, tf)
    assert big["bound"] == "tensor" and big["unit"] == "TFLOP/s"
    assert abs(big["frac"] - big["achieved"] / tf) < 1e-12


def test_engine_names_follow_the_automatic_choice():
    assert bench.engine_of(1, "bf16") == "cluster"
    assert bench.engine_of(32, "q8_0") == "cluster"
    assert bench.engine_of(33, "bf16") == "small"
    assert bench.engine_of(8, "bf16", sampled=True) == "small"
    assert bench.engine_of(40, "bf16") == "small"
    assert bench.engine_of(41, "bf16") == "tile"
    assert bench.engine_of(256, "bf16", sampled=True) == "tile"
