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


class _Opaque:
    """An object a checkpoint must not carry (any pickled class instance)."""

    def __init__(self):
        self.x = 1


def test_checkpoint_loader_refuses_pickled_objects(built_package, tmp_path):
    """load_checkpoint reads with weights_only=True: a file holding a pickled
    class instance is refused before any parameter or state is touched."""
    import pickle

    from adamw_update_gb300.optim import load_checkpoint

    path = tmp_path / "ckpt.pt"
    torch.save({"params": [torch.zeros(3)], "optimizer": {}, "extra": _Opaque()}, path)
    with pytest.raises(pickle.UnpicklingError):
        load_checkpoint(str(path), [torch.ones(3)], None)


def test_checkpoint_extra_must_be_plain_data(built_package):
    from adamw_update_gb300.optim import _check_plain

    _check_plain({"update": 3, "tokens": [1, 2.5, "a", None, (True, b"x")], "t": torch.zeros(2)})
    with pytest.raises(TypeError):
        _check_plain({"update": _Opaque()})
    with pytest.raises(TypeError):
        _check_plain([{1: {2.0}}])  # a set is not plain data here
