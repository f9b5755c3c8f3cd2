"""bench.py's headline line: the numeric digest of the sections it carries
(host logic only, no GPU)."""

import json

import bench


def test_shape_key():
    assert bench._shape_key("M6_N34816_K5120") == "6x34816x5120"


def test_digest_carries_every_row_compactly():
    per = {"M6_N34816_K5120": {"us": 18.0, "weight_GBps": 5282.2}}
    sec = {
        "prefill_w4a8": {"M256_N34816_K5120": {"us": 40.6, "TFLOPs": 2246.4, "frac_fp8_peak": 0.512}},
        "mma_peak_TFLOPs": {"mxf8f6f4_n256": 4383.5, "f8f6f4_n128": 4006.6, "f8f6f4_n256": 4388.3, "mxf4_n256": 8752.5,
                            "sm_mhz": 2070.0},
        "blockfp8": {"M2048_N6144_K2048": {"us": 67.2, "TFLOPs": 766.9, "weight_GBps": 187.2},
                     "M8_N6144_K2048": {"us": 7.3, "TFLOPs": 27.5, "weight_GBps": 1720.4}},
        "skinny_bf16_graph": {"M6_N256_K2048": {"hot_us": 2.834, "pooled_us": 3.011}},
        "quant_per_token": {"M8192_K5120": {"us": 24.87, "GBps": 5060.7}},
        "fused_quant": {"silu_mul_quant_M2048_N17408": {"us": 69.3, "GBps": 2571.8}},
        "w4a4": {"digest": {"decode_GBps": {"6x34816x5120": 4998}}},
        "tiny_w4a8": {"M8_N256_K2048": {"us_quant_plus_gemm": 7.52}},
    }
    d = bench.digest(per, sec, 6777.6)
    assert d["decode_GBps"] == {"6x34816x5120": 5282}
    assert d["prefill_TFLOPs"] == {"256x34816x5120": 2246}
    assert d["prefill_frac"] == {"256x34816x5120": 0.512}
    assert d["blockfp8_TFLOPs_M2048_GBps_else"] == {"2048x6144x2048": 767, "8x6144x2048": 1720}
    assert d["skinny_hot_us"] == {"6x256x2048": 2.834}
    assert d["w4a4"] == {"decode_GBps": {"6x34816x5120": 4998}}
    assert d["mma_peak_TFLOPs"]["mxf4_n256"] == 8752.5
    # the block-FP8 128-token tile's instruction shape (M=128, N=256)
    assert d["mma_peak_TFLOPs"]["f8f6f4_n256"] == 4388.3
    # numbers only, short keys: the full line of the real run stays a few KB
    assert len(json.dumps(d, separators=(",", ":"))) < 1200
