"""Memory and communication ledger of the ZeRO stages (pure Python).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (page title, section):
  [L5] "Lesson 5: ZeRO and FSDP (including the FSDP2 architecture)",
       hpc.payai.win -- section 2 (per-rank memory of stages 0..3 with the
       optimizer's 12 bytes per parameter, and the note on an fp32 gradient
       accumulator), section 3 (communication: one reduce-scatter or one
       all-gather moves (N_d-1)/N_d * Psi per rank; DDP and ZeRO-1/2 move
       2 Psi, ZeRO-3 3 Psi), the worked 7B table that follows section 7.
  [DZ] "Data parallelism and ZeRO memory sharding", jefxiong.cn -- section 3.2
       (16 bytes per parameter: 2 + 2 + 4 + 4 + 4), section 3.3 (the stage
       formulas and the 7.5B / 64-rank example), section 3.4 (reduce-scatter
       + all-gather make the all-reduce), section 4.1 (printed ledgers for
       7.5B/64 and 1.5B/8, decimal GB).
  [ZvF] "ZeRO vs FSDP: memory accounting and communication breakdown for
       large-model distributed training", muhenan.com -- sections 1 and 2
       (16N GB for N billion parameters; 70B on 64 GPUs ~ 17.5 GB).

The memory side is one table: every kind of model state with its bytes per
parameter and the lowest ZeRO stage that partitions it over the ranks.  A
rank holds each kind whole below that stage and a 1/N_d share from it on;
stage 0 is plain data parallelism.  Sizes are in bytes; GB means 1e9 bytes,
as on the pages.
"""
from __future__ import annotations

from collections import namedtuple

StateKind = namedtuple("StateKind", "name bytes_per_param sharded_from_stage")

# Mixed-precision Adam ([DZ] section 3.2; [L5] section 2): the low-precision
# parameters are partitioned by stage 3, the low-precision gradients by
# stage 2, and the fp32 optimizer state (master weights, m, v: 4 + 4 + 4) by
# stage 1.
MODEL_STATE = (
    StateKind("parameters", 2, 3),
    StateKind("gradients", 2, 2),
    StateKind("optimizer", 12, 1),
)
# An fp32 gradient accumulator for micro-batching follows the gradients: whole
# while they are whole (stages 0 and 1), partitioned with them from stage 2
# ([L5] section 2, note).
FP32_ACCUMULATOR = StateKind("fp32 accumulator", 4, 2)

KIND_BYTES = {k.name: k.bytes_per_param for k in MODEL_STATE + (FP32_ACCUMULATOR,)}
STAGES = (0, 1, 2, 3)


def _require(psi, n):
    if not (psi > 0 and n > 0):
        raise ValueError(f"ledger needs psi > 0 and n > 0 (got psi={psi!r}, n={n!r})")


def _require_stage(stage):
    if stage not in STAGES:
        raise ValueError(f"no ZeRO stage {stage!r}: use 0 (replicated) to 3")


def held_fraction(kind: StateKind, n: int, stage: int) -> float:
    """The share of one state kind a rank keeps: all of it below the stage that
    partitions it, 1/n from that stage on."""
    return 1.0 / n if stage >= kind.sharded_from_stage else 1.0


def per_rank_state_bytes(psi: float, n: int, stage: int, accumulator: bool = False) -> float:
    """Model-state bytes one of n ranks holds for psi parameters under a ZeRO
    stage ([L5] section 2; [DZ] section 3.3): the sum over the state table of
    bytes per parameter x psi x the share the rank keeps."""
    _require(psi, n)
    _require_stage(stage)
    kinds = MODEL_STATE + ((FP32_ACCUMULATOR,) if accumulator else ())
    return sum(k.bytes_per_param * psi * held_fraction(k, n, stage) for k in kinds)


def bytes_per_param(n: int, stage: int) -> float:
    """Per-rank model-state bytes divided by the parameter count."""
    return per_rank_state_bytes(1.0, n, stage)


def memory_saving(n: int, stage: int) -> float:
    """How many times smaller the per-rank state is than plain data parallel."""
    return per_rank_state_bytes(1.0, n, 0) / per_rank_state_bytes(1.0, n, stage)


def collective_volume(psi: float, n: int) -> float:
    """Elements each rank moves in one reduce-scatter or one all-gather of Psi
    elements over n ranks (ring model, [L5] section 3; [DZ] section 3.4)."""
    _require(psi, n)
    return (n - 1) / n * psi


# Collectives of one training step per stage ([L5] section 3): an all-reduce
# is a reduce-scatter plus an all-gather; ZeRO-1/2 reduce-scatter the
# gradients and all-gather the updated parameters; ZeRO-3 also all-gathers the
# parameters a second time for the backward pass.
COLLECTIVES_PER_STEP = {0: 2, 1: 2, 2: 2, 3: 3}


def comm_elements(psi: float, n: int, stage: int, exact: bool = True) -> float:
    """Elements moved per rank per training step.  exact=False takes each
    collective as a full Psi, the pages' large-n forms 2 Psi and 3 Psi."""
    _require(psi, n)
    _require_stage(stage)
    per_collective = collective_volume(psi, n) if exact else psi
    return COLLECTIVES_PER_STEP[stage] * per_collective


def comm_bytes(psi: float, n: int, stage: int, exact: bool = False,
               bytes_per_element: int = KIND_BYTES["gradients"]) -> float:
    """Bytes per rank per step; the pages count 2-byte (bf16/fp16) elements."""
    return comm_elements(psi, n, stage, exact=exact) * bytes_per_element


def adam_scalars_per_rank(psi: int, n: int, sharded: bool) -> int:
    """Number of Adam m and v scalars a rank holds ([DZ] section 4.2)."""
    if not sharded:
        return 2 * psi
    if psi % n:
        raise ValueError(f"{n} shards do not divide {psi} parameters evenly")
    return 2 * (psi // n)


def gb(nbytes: float) -> float:
    """Decimal gigabytes, the unit the pages use ([DZ] section 3.3)."""
    return nbytes / 1e9


StageLedger = namedtuple("StageLedger", "stage state_gb bytes_per_param saving_vs_ddp comm_gb")


def ledger_rows(psi: float, n: int):
    """One StageLedger per stage 0..3 for psi parameters on n ranks: the
    per-rank model state in GB and per parameter, the saving against plain
    data parallel, and the approximate communication per step in GB (the
    quantities [DZ] section 4.1 prints)."""
    return [StageLedger(stage=s, state_gb=gb(per_rank_state_bytes(psi, n, s)),
                        bytes_per_param=bytes_per_param(n, s),
                        saving_vs_ddp=memory_saving(n, s),
                        comm_gb=gb(comm_bytes(psi, n, s, exact=False)))
            for s in STAGES]
