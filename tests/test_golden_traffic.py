"""The byte model behind the roofline fractions reproduces the traffic the
pages print (Table 2 of §5.2 and the 21 GB / 42 GB figure of §1)."""
import json
import os

from late_interaction_retrieval_maxsim_gb300 import roofline

GOLD = os.path.join(os.path.dirname(__file__), "golden", "traffic_table.json")


def test_table2_naive_and_fused_bytes():
    g = json.load(open(GOLD))
    for row in g["rows"]:
        naive = roofline.naive_hbm_bytes(g["n_docs"], row["lq"], row["ld"], g["dim"]) / 1e9
        fused = roofline.fused_input_bytes(g["n_docs"], row["ld"], g["dim"]) / 1e9
        assert round(naive, 2) == row["naive_gb"], row
        assert round(fused, 2) == row["fused_gb"], row
        assert round(naive / fused) == row["ratio"], row


def test_materialised_tensor_size():
    m = json.load(open(GOLD))["materialised"]
    assert round(roofline.materialised_tensor_bytes(m["n_docs"], m["lq"], m["ld"], 2) / 1e9) == m["fp16_gb"]
    assert round(roofline.materialised_tensor_bytes(m["n_docs"], m["lq"], m["ld"], 4) / 1e9) == m["fp32_gb"]


def test_flops_of_colpali_floor():
    """1K ColPali pairs are 2*1024*1024*128*1000 = 2.68e11 FLOP (the pages'
    'matmul arithmetic floor' of §5.2 is this count at the A100's rate)."""
    assert roofline.forward_flops(1024, 1000 * 1024) == 2 * 128 * 1024 * 1024 * 1000
