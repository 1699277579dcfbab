"""Integer contracts against the worked examples the pages print."""
import json
import os

import pytest

from oracle import contracts

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "contracts.json")))


@pytest.mark.parametrize("case", GOLDEN["data_parallel"], ids=lambda c: c["cite"][:40])
def test_data_parallel_size(case):
    assert contracts.data_parallel_size(case["world"], case["tp"], case["pp"], case["cp"],
                                        case["ep"]) == case["dp"]


def test_data_parallel_size_rejects_remainder():
    with pytest.raises(ValueError):
        contracts.data_parallel_size(64, 4, 4, 3)


@pytest.mark.parametrize("case", GOLDEN["global_batch"], ids=lambda c: c["cite"][:40])
def test_global_batch(case):
    assert contracts.global_batch(case["micro_batch"], case["dp"], case["accum"]) == case["global_batch"]
    assert contracts.grad_accum_steps(case["global_batch"], case["micro_batch"], case["dp"]) == case["accum"]


def test_grad_accum_rejects_remainder():
    with pytest.raises(ValueError):
        contracts.grad_accum_steps(30, 4, 2)


@pytest.mark.parametrize("case", GOLDEN["tp_divisible"], ids=lambda c: c["cite"][:40])
def test_tp_divisible(case):
    assert contracts.tp_divisible(case["hidden"], case["heads"], case["tp"]) == case["ok"]
    if case["ok"]:
        assert [case["hidden"] // case["tp"], case["heads"] // case["tp"]] == case["per_part"]


@pytest.mark.parametrize("case", GOLDEN["pp_layers"], ids=lambda c: c["cite"][:40])
def test_pp_layers(case):
    assert contracts.pp_layers_ok(case["layers"], case["pp"]) == case["ok"]


@pytest.mark.parametrize("case", GOLDEN["model_state_bytes"], ids=lambda c: str(c["dp"]))
def test_model_state_bytes(case):
    assert contracts.model_state_bytes_per_param(case["dp"]) == case["bytes_per_param"]


@pytest.mark.parametrize("case", GOLDEN["bf16_weights"], ids=lambda c: str(c["params"]))
def test_bf16_weight_bytes(case):
    assert contracts.bf16_weight_bytes(case["params"]) == case["bytes"]
