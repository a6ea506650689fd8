"""Host logic of the FP8 linear layer: the autocast scope's recipe stack."""
import pytest

from scaled_quantize_gemm_amax_gb300 import linear as L


def test_fp8_autocast_scopes_nest():
    assert isinstance(L.get_fp8_recipe(), L.Float8CurrentScaling)
    with L.fp8_autocast(fp8_recipe=L.Float8BlockScaling()):
        assert isinstance(L.get_fp8_recipe(), L.Float8BlockScaling)
        with L.fp8_autocast(fp8_recipe=L.MXFP8BlockScaling()):
            assert isinstance(L.get_fp8_recipe(), L.MXFP8BlockScaling)
        with L.fp8_autocast(enabled=False):
            assert isinstance(L.get_fp8_recipe(), L.Float8BlockScaling)
        assert isinstance(L.get_fp8_recipe(), L.Float8BlockScaling)
    assert isinstance(L.get_fp8_recipe(), L.Float8CurrentScaling)


def test_recipe_operand_kinds():
    R = L.Recipe
    assert L._kinds(L.Float8CurrentScaling()) == (R.TENSOR, R.TENSOR)
    assert L._kinds(L.Float8DelayedScaling()) == (R.TENSOR, R.TENSOR)
    assert L._kinds(L.Float8BlockScaling()) == (R.BLOCK_1x128, R.BLOCK_128x128)
    assert L._kinds(L.MXFP8BlockScaling()) == (R.MX_1x32_TILED, R.MX_1x32_TILED)
    with pytest.raises(TypeError):
        L._kinds(object())
