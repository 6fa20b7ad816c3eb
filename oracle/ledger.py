"""Memory and communication ledger of the ZeRO stages (pure Python).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (page title, section):
  [L5] "Lesson 5: ZeRO and FSDP (including the FSDP2 architecture)",
       hpc.payai.win -- section 2 (per-rank memory M0..M3 with the optimizer
       multiplier k = 12 and the fp32 gradient-accumulation note), section 3
       (communication: V_RS = V_AG = (N_d-1)/N_d * Psi; DDP 2 Psi; ZeRO-1/2
       2 Psi; ZeRO-3 3 Psi), the worked 7B table that follows section 7.
  [DZ] "Data parallelism and ZeRO memory sharding", jefxiong.cn -- section 3.2
       (16 bytes per parameter: 2 + 2 + 4 + 4 + 4), section 3.3 (the three
       stage formulas and the 7.5B / 64-rank example), section 3.4
       (reduce-scatter + all-gather make the all-reduce), section 4.1 (printed
       ledgers for 7.5B/64 and 1.5B/8, decimal GB).
  [ZvF] "ZeRO vs FSDP: memory accounting and communication breakdown for
       large-model distributed training", muhenan.com -- sections 1 and 2
       (16N GB for N billion parameters; 70B on 64 GPUs ~ 17.5 GB).

Sizes are in bytes; GB means 1e9 bytes, as on the pages.
"""
from __future__ import annotations

# Bytes per parameter of each model-state kind under bf16/fp16 mixed-precision
# Adam ([DZ] section 3.2).
PARAM_BYTES = 2          # low-precision parameters
GRAD_BYTES = 2           # low-precision gradients
MASTER_BYTES = 4         # fp32 master weights
MOMENT_BYTES = 4         # each of Adam's m and v
OPTIMIZER_MULTIPLIER = MASTER_BYTES + 2 * MOMENT_BYTES   # k = 12 ([L5] section 2)
FP32_ACCUM_BYTES = 4     # fp32 gradient accumulator ([L5] section 2, note)

STAGES = (0, 1, 2, 3)    # 0 = plain data parallel (DDP)


def _check(psi, n):
    if psi <= 0 or n <= 0:
        raise ValueError("parameter count and rank count must be positive")


def model_state_bytes(psi: float, n: int, stage: int, k: float = OPTIMIZER_MULTIPLIER,
                      fp32_grad_accum: bool = False) -> float:
    """Per-rank model-state bytes for ZeRO stage 0..3 ([L5] section 2).

    stage 0: 2Psi + 2Psi + k Psi                 (everything replicated)
    stage 1: 2Psi + 2Psi + k Psi / n             (optimizer state sharded)
    stage 2: 2Psi + (2Psi + k Psi) / n           (+ gradients sharded)
    stage 3: (2Psi + 2Psi + k Psi) / n           (+ parameters sharded)
    The optional fp32 accumulator is replicated for stages 0 and 1 (+4 Psi)
    and sharded for stages 2 and 3 (+4 Psi / n).
    """
    _check(psi, n)
    if stage not in STAGES:
        raise ValueError("stage must be 0..3")
    params = PARAM_BYTES * psi
    grads = GRAD_BYTES * psi
    optim = k * psi
    if stage == 0:
        total = params + grads + optim
    elif stage == 1:
        total = params + grads + optim / n
    elif stage == 2:
        total = params + (grads + optim) / n
    else:
        total = (params + grads + optim) / n
    if fp32_grad_accum:
        total += FP32_ACCUM_BYTES * psi if stage <= 1 else FP32_ACCUM_BYTES * psi / n
    return total


def bytes_per_param(n: int, stage: int) -> float:
    """Per-rank model-state bytes divided by the parameter count."""
    return model_state_bytes(1.0, n, stage)


def memory_saving(n: int, stage: int) -> float:
    """How many times smaller the per-rank state is than plain data parallel."""
    return model_state_bytes(1.0, n, 0) / model_state_bytes(1.0, n, stage)


def collective_volume(psi: float, n: int) -> float:
    """Elements each rank moves in one reduce-scatter or one all-gather of Psi
    elements over n ranks (ring model, [L5] section 3; [DZ] section 3.4)."""
    _check(psi, n)
    return (n - 1) / n * psi


def comm_elements(psi: float, n: int, stage: int, exact: bool = True) -> float:
    """Elements moved per rank per training step ([L5] section 3).

    stage 0: all-reduce = reduce-scatter + all-gather
    stage 1/2: reduce-scatter of gradients + all-gather of updated parameters
    stage 3: forward all-gather + backward all-gather + reduce-scatter
    exact=False gives the pages' large-n approximations 2 Psi and 3 Psi.
    """
    _check(psi, n)
    if stage not in STAGES:
        raise ValueError("stage must be 0..3")
    one = collective_volume(psi, n) if exact else psi
    if stage in (0, 1, 2):
        return 2 * one
    return 3 * one


def comm_bytes(psi: float, n: int, stage: int, exact: bool = False,
               bytes_per_element: int = GRAD_BYTES) -> float:
    """Bytes per rank per step; the pages count 2-byte (bf16/fp16) elements."""
    return comm_elements(psi, n, stage, exact=exact) * bytes_per_element


def adam_scalars_per_rank(psi: int, n: int, sharded: bool) -> int:
    """Number of Adam m and v scalars a rank holds ([DZ] section 4.2)."""
    if sharded:
        if psi % n:
            raise ValueError("the shard count must divide the parameter count")
        return 2 * (psi // n)
    return 2 * psi


def gb(nbytes: float) -> float:
    """Decimal gigabytes, the unit the pages use ([DZ] section 3.3)."""
    return nbytes / 1e9


def ledger_rows(psi: float, n: int):
    """Rows (stage, bytes/param, state GB, saving vs DDP, comm GB per step) in
    the layout of the printed ledgers of [DZ] section 4.1 (approximate comm)."""
    rows = []
    for stage in STAGES:
        rows.append((stage, bytes_per_param(n, stage), gb(model_state_bytes(psi, n, stage)),
                     memory_saving(n, stage), gb(comm_bytes(psi, n, stage, exact=False))))
    return rows
