"""The benchmark's work model (the algorithmic bytes and flops its roofline
fractions divide by), on the CPU: a hand-counted single matrix, and the
GPT-2 XL totals that the measured results are quoted against."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402


def test_work_model_single_matrix_by_hand():
    # 768 x 768 fp32 matrix, B = 4 (k = 192), 1024 fp32 tokens.
    # update: G read 4 B, M read + write 8 B, W read + write 8 B per entry,
    # plus the four 192 x 192 fp32 bases read once
    wm = bench.work_model([(768, 768)], 4, 1024, pbytes=4, xbytes=4)
    assert wm["update_bytes"] == 768 * 768 * 20 + 4 * 4 * 192 * 192 == 12_386_304
    # projection and reconstruction: 2 k flops per entry each
    assert wm["update_flops"] == 2 * 2 * 192 * 768 * 768 == 452_984_832
    # moments: X read once (fp32), four blocks of A read and written
    assert wm["acc_bytes"] == 4 * 1024 * 768 + 8 * 4 * 192 * 192 == 4_325_376
    # symmetric block products: N k (k + 1) multiply-adds counted as flops per block
    assert wm["acc_flops"] == 4 * 1024 * 192 * 193
    # eigendecomposition with vectors: 9 k^3 per block
    assert wm["refresh_flops"] == 9 * 4 * 192 ** 3 == 254_803_968


def test_work_model_gpt2_xl_totals():
    shapes, _ = bench.model_shapes("gpt2-xl")
    assert len(shapes) == 289
    params = sum(m * n for m, n in shapes)
    # per layer q, k, v, o (1600 x 1600), fc (6400 x 1600), proj (1600 x 6400); embedding
    assert params == 48 * (4 * 1600 * 1600 + 2 * 6400 * 1600) + 50257 * 1600 == 1_554_971_200
    wm = bench.work_model(shapes, 16, 8192, pbytes=2, xbytes=2)
    # per layer 5 matrices of input width 1600 (k = 100) and one of 6400
    # (k = 400), 48 layers, plus the 50257 x 1600 embedding (k = 100)
    blocks_k3 = 48 * (5 * 16 * 100 ** 3 + 16 * 400 ** 3) + 16 * 100 ** 3
    assert wm["refresh_flops"] == 9 * blocks_k3 == 477_072_000_000
    assert wm["update_bytes"] == 14 * params + 4 * sum(n * (n // 16) for _, n in shapes)
    assert wm["update_bytes"] == 22_415_356_800
    assert wm["update_flops"] == 1_211_812_480_000
    assert wm["acc_bytes"] == 12_642_355_200


def test_work_model_orthogonal_iteration_and_output_side():
    # one step: 2 k^3 (A Q) + k^3 (Gram) + k^3 / 3 (Cholesky) + k^3 (solve)
    wm = bench.work_model([(64, 192)], 2, 0, refresh="orth", orth_steps=1)
    assert abs(wm["refresh_flops"] - 2 * 96 ** 3 * 13 / 3) < 1e-6
    # Dobb-G: the same work as Dobb on the transposed problem
    a = bench.work_model([(384, 256)], 2, 512, sides=["output"])
    b = bench.work_model([(256, 384)], 2, 512)
    assert a == b
