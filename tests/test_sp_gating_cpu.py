"""The host-side sharding gate for sequence-parallel MLPs (prhub analysis of vllm PR
#50656, section "实现拆解", item 2: shard only when the opt-in switch is on, the
model runs sequence-parallel, the call site is eligible, tp > 1 and both hidden and
intermediate sizes divide by tp; otherwise stay replicated).  Its six cases are the
branches that section lists for the gating test: opt-in, not sequence-parallel, the
FusedMoE path not eligible, tp = 1 and 6144 % 5 != 0, plus the default (switch off).
No GPU is needed: the gate is a pure host function of the library."""
import pytest

import moe_shared_expert_gb300 as mse
from moe_shared_expert_gb300 import _build

H, I = 7168, 6144      # Kimi-K3 shared expert: hidden 7168, shared intermediate 6144


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    mse.lib()


@pytest.mark.parametrize("enabled,use_sp,eligible,tp,expect", [
    (True, True, True, 4, True),      # opted in, sequence-parallel, eligible call site: shard
    (False, True, True, 4, False),    # the switch is off by default: replicate
    (True, False, True, 4, False),    # no sequence parallelism: the ordinary TP path, not this gate
    (True, True, False, 4, False),    # shared experts on the FusedMoE path are not eligible
    (True, True, True, 1, False),     # nothing to shard over
    (True, True, True, 5, False),     # 6144 % 5 != 0: fall back to replication, no error
], ids=["opt_in", "default_off", "not_sp", "fused_moe_not_eligible", "tp1", "not_divisible"])
def test_gate_cases(enabled, use_sp, eligible, tp, expect):
    assert mse.shard_sequence_parallel_mlp(enabled, use_sp, eligible, tp, H, I) is expect


@pytest.mark.parametrize("tp", [2, 4, 8, 16])
def test_gate_shards_at_the_tp_sizes_of_the_tuned_shapes(tp):
    # TP4/TP8/TP16 are the sharded shapes the pages' tuned GEMM table lists
    assert mse.shard_sequence_parallel_mlp(True, True, True, tp, H, I)


def test_gate_needs_both_sizes_divisible():
    assert 6144 % 3 == 0 and 7168 % 3 != 0
    assert not mse.shard_sequence_parallel_mlp(True, True, True, 3, H, I)     # hidden fails
    assert 7168 % 7 == 0 and 6144 % 7 != 0
    assert not mse.shard_sequence_parallel_mlp(True, True, True, 7, H, I)     # intermediate fails
    assert mse.shard_sequence_parallel_mlp(True, True, True, 3, 768, 384)    # both divide
    assert not mse.shard_sequence_parallel_mlp(True, True, True, 0, H, I)
    assert not mse.shard_sequence_parallel_mlp(True, True, True, -4, H, I)

