"""Model-state memory and communication ledger (TEST INFRASTRUCTURE ONLY).

Sources (page title, section):
  "Learn: ZeRO & FSDP", section 3: per parameter 2 B bf16 weights + 2 B bf16
      gradients + K = 12 B of fp32 optimizer state (master, m, v) = 16 B.
  "Learn: ZeRO & FSDP", section 4: per-GPU model state for N_d ranks,
      DDP (2+2+K)Psi; ZeRO-1 4Psi + K Psi/N_d; ZeRO-2 2Psi + (2+K)Psi/N_d;
      ZeRO-3 (2+2+K)Psi/N_d.  Communication: DDP = ZeRO-1 = ZeRO-2 = 2Psi,
      ZeRO-3 = 3Psi elements per step.
  "ZeRO and FSDP sharding", How it works: 16Psi/N bytes per GPU under ZeRO-3,
      3Psi communicated elements per step (1.5x DDP).
"""
K_ADAM = 12  # fp32 master + m + v, bytes per parameter


def model_state_bytes(psi: float, n_d: int, stage: int, k: int = K_ADAM) -> float:
    """Per-GPU model-state bytes at ZeRO stage 0 (DDP), 1, 2 or 3."""
    if stage == 0:
        return (2 + 2 + k) * psi
    if stage == 1:
        return 2 * psi + 2 * psi + k * psi / n_d
    if stage == 2:
        return 2 * psi + (2 + k) * psi / n_d
    if stage == 3:
        return (2 + 2 + k) * psi / n_d
    raise ValueError(f"stage {stage}")


def comm_elements(psi: float, stage: int) -> float:
    """Elements communicated per step (before the ring's (N-1)/N factor)."""
    if stage in (0, 1, 2):
        return 2 * psi  # reduce-scatter Psi + all-gather Psi = one all-reduce
    if stage == 3:
        return 3 * psi  # all-gather (forward) + all-gather (backward) + reduce-scatter
    raise ValueError(f"stage {stage}")


def min_ranks_to_fit(psi: float, hbm_bytes: float, stage: int, k: int = K_ADAM):
    """Smallest N_d whose per-GPU model state fits in hbm_bytes, or None if none does."""
    for n in range(1, 1 << 20):
        if model_state_bytes(psi, n, stage, k) <= hbm_bytes:
            return n
        if stage in (1, 2) and model_state_bytes(psi, 1 << 40, stage, k) > hbm_bytes:
            return None  # the replicated floor alone does not fit
    return None
