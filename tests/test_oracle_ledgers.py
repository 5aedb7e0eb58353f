"""Pins of split bounds, owner grids and byte ledgers (M4.5 §0x03A-§0x03G, M8.6 §0x04B)."""

from oracle import quant
from oracle import split_state as ss
from tests.conftest import golden

MiB = 1 << 20


def test_balanced_split_lengths():
    g = golden("split_ledgers.json")
    for T, lens in g["split_lengths"].items():
        b = ss.balanced_split_bounds(int(T), g["call"]["S"])
        assert [e - a for a, e in b] == lens
        assert b[0][0] == 0 and b[-1][1] == int(T)
        assert all(b[i][1] == b[i + 1][0] for i in range(len(b) - 1))


def test_fixed_chunk_policy_covers_exactly():
    for T in (0, 1, 63, 64, 65, 3587):
        ch = ss.fixed_chunk_bounds(T, 64)
        assert len(ch) == -(-T // 64)
        assert sum(e - a for a, e in ch) == T


def test_owner_counts():
    g = golden("split_ledgers.json")
    c = g["call"]
    assert ss.owner_counts(c["B"], c["H_q"], c["S_cap"]) == g["owners"]


def test_workspace_and_reduction_bytes():
    g = golden("split_ledgers.json")
    c = g["call"]
    n = c["B"] * c["H_q"] * c["S"]
    w = g["workspace"]
    assert ss.workspace_mlu_bytes(1, c["d"]) == w["mlu_bytes_per_state"]
    assert ss.workspace_mlu_bytes(n, c["d"]) == w["mlu_total"]
    assert ss.workspace_lse_o_bytes(1, c["d"]) == w["lse_o_bytes_per_state"]
    assert ss.workspace_lse_o_bytes(n, c["d"]) == w["lse_o_total"]
    r = g["reduction_path"]
    assert ss.reduction_path_bytes(w["mlu_total"], c["B"], c["H_q"], c["d"]) == r["mlu"]
    assert ss.reduction_path_bytes(w["lse_o_total"], c["B"], c["H_q"], c["d"]) == r["lse_o"]


def test_kv_ledgers():
    g = golden("split_ledgers.json")
    c = g["call"]
    k = g["kv_ledgers"]
    uniq = ss.kv_unique_bytes(c["T"], c["H_kv"], c["d"], c["d"], c["b_cache"])
    dem = ss.kv_qhead_demand_bytes(c["T"], c["H_q"], c["d"], c["d"], c["b_cache"])
    assert uniq == k["kv_unique"] and dem == k["kv_qhead_demand"]
    q_unique = c["B"] * c["H_q"] * c["d"] * 2
    assert q_unique == k["q_unique"] and q_unique * c["S"] == k["q_demand_every_split"]
    red = g["reduction_path"]
    assert dem + k["q_demand_every_split"] + red["mlu"] == k["mlu_full_demand"]
    assert dem + k["q_demand_every_split"] + red["lse_o"] == k["lse_o_full_demand"]


def test_capacity_envelope_fixture():
    g = golden("split_ledgers.json")["capacity_fixture"]
    r = ss.capacity_envelope(g["T"], g["S"], g["S_cap"], g["H_q"])
    for key in ("producers", "active", "identity", "reducers"):
        assert r[key] == g[key]
    assert r["split_lengths"][0][:g["S"]] == g["request0_lengths"]
    assert r["split_lengths"][1][:g["S"]] == [0] * g["S"]


def test_head_width_tail():
    g = golden("split_ledgers.json")["head_width"]
    assert ss.padded_width(g["d_v"], g["align"]) == g["d_v_padded"]
    n = g["logical_bytes"] // ss.workspace_mlu_bytes(1, g["d_v"])
    assert ss.workspace_mlu_bytes(n, g["d_v"]) == g["logical_bytes"]
    assert ss.workspace_mlu_bytes(n, g["d_v_padded"]) == g["capacity_bytes"]


def test_int2_kivi_like_ledger():
    g = golden("kv_ledger.json")
    s = g["shape"]
    r = quant.served_bytes(**s)
    for key, mib in g["MiB"].items():
        k = {"codes": "codes", "k_qparams": "k_qparams", "v_qparams": "v_qparams",
             "residual": "residual", "total": "total"}[key]
        assert r[k] == mib * MiB
