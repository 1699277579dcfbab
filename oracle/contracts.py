"""Integer contracts of the Megatron parallel layout, as the pages state them.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).  Pure integer arithmetic;
pinned by the worked examples in ``tests/golden/contracts.json``.
"""
from __future__ import annotations


def data_parallel_size(world: int, tp: int, pp: int, cp: int = 1, ep: int = 1) -> int:
    """DP from ``world = TP x PP x CP x EP x DP``.

    ai.lansai.wang/82226.html, section 并行度先做整数校验 (dense models, EP = 1 in
    the worked example).  Raises ValueError when the product does not divide.
    """
    model = tp * pp * cp * ep
    if model <= 0 or world % model:
        raise ValueError(f"world size {world} not divisible by TP*PP*CP*EP = {model}")
    return world // model


def grad_accum_steps(global_batch: int, micro_batch: int, dp: int) -> int:
    """Accumulation steps from ``global = micro x DP x accum``.

    cf-1.com/news/5344657, section 2.1 (数据并行) and the section 4.1 command.
    """
    per_step = micro_batch * dp
    if per_step <= 0 or global_batch % per_step:
        raise ValueError(f"global batch {global_batch} not divisible by micro*DP = {per_step}")
    return global_batch // per_step


def global_batch(micro_batch: int, dp: int, accum: int) -> int:
    return micro_batch * dp * accum


def tp_divisible(hidden: int, heads: int, tp: int, ffn: int | None = None,
                 vocab: int | None = None) -> bool:
    """True when every tensor-parallel-split dimension divides by ``tp``.

    cf-1.com/news/5344657, section 2.2: hidden size, head count (and vocab)
    must divide by the TP degree.
    """
    dims = [hidden, heads] + [v for v in (ffn, vocab) if v is not None]
    return tp >= 1 and all(v % tp == 0 for v in dims)


def pp_layers_ok(num_layers: int, pp: int) -> bool:
    """cf-1.com/news/5344657, section 2.3: num_layers % PP must be 0."""
    return pp >= 1 and num_layers % pp == 0


def model_state_bytes_per_param(dp: int | None = None) -> float:
    """Bytes of model state per parameter (bf16 params, fp32 main grads, Adam).

    ai.lansai.wang/82226.html, section 分布式优化器能省多少内存: 18 without the
    distributed optimizer, 6 + 12/d with it (d = data-parallel size).
    """
    if dp is None:
        return 18.0
    return 6.0 + 12.0 / dp


def bf16_weight_bytes(params: int) -> int:
    """cf-1.com/news/5344657, section 1.1: 2 bytes per bf16 parameter."""
    return 2 * params
