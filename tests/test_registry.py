"""The kernel registry: what an ordinary run gets, and how a variant is
selected (no GPU needed)."""
import pytest

from w4a16_int4_weight_gemv_gb300 import registry


def test_shipped_defaults_are_pinned(monkeypatch):
    # an ordinary run (no selection in the environment) gets the fast paths
    monkeypatch.delenv(registry.ENV, raising=False)
    assert registry.selection() == {"w4a16_dense": "planned", "w4a16_grouped": "planned",
                                    "w3a16_grouped": "fp16_mma", "w4a16_ffn": "fused",
                                    "w3a16_ffn": "fp16_mma"}
    for op, var in registry.DEFAULTS.items():
        assert registry.get(op) is registry.OPS[op][var]


def test_every_default_is_registered():
    assert set(registry.DEFAULTS) == set(registry.OPS)
    for op, var in registry.DEFAULTS.items():
        assert var in registry.OPS[op]
        assert all(callable(f) for f in registry.OPS[op].values())


def test_environment_selects_a_variant(monkeypatch):
    monkeypatch.setenv(registry.ENV, "w4a16_dense=warp_mma, w4a16_ffn=chain")
    sel = registry.selection()
    assert sel["w4a16_dense"] == "warp_mma" and sel["w4a16_ffn"] == "chain"
    assert sel["w4a16_grouped"] == "planned"
    assert registry.get("w4a16_dense") is registry.OPS["w4a16_dense"]["warp_mma"]


@pytest.mark.parametrize("text", ["w4a16_dense=fastest", "w4a16_gemm=planned", "w4a16_dense"])
def test_unknown_names_are_rejected(text):
    with pytest.raises(ValueError):
        registry.selection(text)


def test_variants_list_matches_table():
    assert registry.variants("w4a16_dense") == ["planned", "cuda_core", "warp_mma", "tcgen05",
                                                "fp16_mma"]
    assert registry.variants("w4a16_grouped") == ["planned", "tma", "fp16_mma"]
