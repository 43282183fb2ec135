"""Values the pages print, kept as small cited fixtures under tests/golden/,
against the constants and workloads that rest on them (CPU)."""
import os

import bench
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].split()
            for key, val in zip(line[::2], line[1::2]):
                vals[key] = float(val)
    return vals


def test_nominal_peaks_are_the_pages():
    g = _read("b200_dense_peaks.txt")
    assert bench.NOMINAL_TFLOPS["bf16"] == g["bf16_dense_pflops"] * 1000
    assert bench.NOMINAL_TFLOPS["fp8"] == g["fp8_dense_pflops"] * 1000


def test_token_grids_follow_the_latent_table():
    g = _read("flux_dev_latent_1024.txt")
    px_per_token = g["resolution"] / g["latent_h"]
    assert px_per_token == g["resolution"] / g["latent_w"] == 16
    w1 = synthetic.WORKLOADS["flux_1024_4608"]
    assert (w1.img_h, w1.img_w) == (g["latent_h"], g["latent_w"])
    assert w1.tokens == w1.txt_len + 64 * 64
    for name in ("flux_2048_16896", "fp8_cfg_2048_16896"):
        w = synthetic.WORKLOADS[name]
        assert (w.img_h, w.img_w) == (2048 / px_per_token, 2048 / px_per_token)
    i2i = synthetic.WORKLOADS["i2i_2048_33280"]
    assert (i2i.img_h, i2i.img_w, i2i.ref_h, i2i.ref_w) == (128, 128, 128, 128)
