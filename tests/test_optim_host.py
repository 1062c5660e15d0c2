"""PackedAdamW's argument checks, on the CPU (no kernel runs): the execution
contract of "Packed AdamW / Reference / v1.0.0" -- contiguous CUDA FP32
parameters on one device, one parameter group."""
import pytest
import torch


def test_rejects_what_the_contract_excludes(built_package):
    from adamw_update_gb300.optim import PackedAdamW

    with pytest.raises(ValueError):
        PackedAdamW([torch.nn.Parameter(torch.zeros(4))])  # not on a CUDA device
    with pytest.raises(ValueError):
        PackedAdamW([torch.nn.Parameter(torch.zeros(4))], mode="int8")
    with pytest.raises(ValueError):
        PackedAdamW([torch.nn.Parameter(torch.zeros(4))], betas=(1.0, 0.999))
    with pytest.raises(ValueError):
        PackedAdamW([{"params": [torch.nn.Parameter(torch.zeros(2))]},
                     {"params": [torch.nn.Parameter(torch.zeros(2))]}])
