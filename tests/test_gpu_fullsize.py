"""Full-size parity, in the launch configuration bench.py times: each
workload runs at its full size (the paged pools of the benchmark, tens to a
hundred GB of HBM) through the same code as the benchmark, and random sampled
outputs are recomputed one by one by the fp64 oracle (copies bit-exact,
rotated / patched values within 1 bf16 ulp).  Smaller cases with full-pool
comparison live in the other GPU test files."""
import types

import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _run(workload: str) -> dict:
    args = types.SimpleNamespace(steps=2, warmup=3, check=True, small=False,
                                 no_cpu_baseline=True, gpus=1, impl="ours", workload=workload)
    return bench.WORKLOADS[workload](args, 0, 1, 0)


def _assert_clean(sample: dict, what: str):
    assert sample, f"{what}: no parity sample"
    for k, v in sample.items():
        if k.endswith("beyond") or k.endswith("differing"):
            assert v == 0, f"{what}: {k} = {v} ({sample})"


@pytest.mark.parametrize("workload", ["relocate-mla", "splice-mla-128k", "relocate-gqa-patch",
                                      "relocate-mla-patch", "splice-mla-128k-composed",
                                      "splice-mla-128k-remap", "window-gqa", "cdc-tokens",
                                      "families"])
def test_full_size_sampled_parity(workload):
    out = _run(workload)
    _assert_clean(out["parity_sample"], workload)
    assert out["gpu_launches"] > 0


def test_sweep_every_point_sampled_parity():
    out = _run("sweep-mla")
    cfg = out["config"]
    for part in ("relocate", "splice", "patch"):
        for pt in cfg[part]:
            _assert_clean(pt["parity_sample"], f"sweep {part} {pt}")
    assert len(cfg["relocate"]) == 30
