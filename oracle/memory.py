"""Model-state memory per GPU, in bytes, for plain data parallelism and the
three ZeRO stages.  TEST INFRASTRUCTURE ONLY (part of the oracle).

Mixed-precision Adam keeps, per parameter: a half-precision parameter (2
bytes), a half-precision gradient (2 bytes) and K = 12 bytes of optimizer
state (fp32 master weight, momentum and variance).  ZeRO partitions these
among N_d data-parallel ranks:

* "ZeRO 技术原理：基础与实现" (jianzhnie.github.io), section 3 "为什么需要 ZeRO"
  ((2 + 2 + K) Psi = 16 Psi) and 3.1.1-3.1.3 (the three stages);
* "千亿参数模型如何塞进有限显卡：ZeRO如何用分片消除数据并行的内存冗余"
  (answer.freetools.me), "Stage 1：优化器状态分片", "Stage 2：梯度分片",
  "Stage 3：参数分片" (4 Psi + 12 Psi / N_d, 2 Psi + 14 Psi / N_d, 16 Psi / N_d);
* "DeepSpeed ZeRO" (formulaic.cloudchewie.com), the memory tables of
  "ZeRO Stage 1" and "ZeRO Stage 2" ((2 + 2 + K/N_d) Phi, (2 + (2 + K)/N_d) Phi).
"""
from __future__ import annotations

from fractions import Fraction

HALF_PARAM_BYTES = 2
HALF_GRAD_BYTES = 2
K_ADAM_MIXED = 12  # fp32 master + momentum + variance


def plain_dp(psi, k=K_ADAM_MIXED):
    """Every rank holds all model states: (2 + 2 + K) Psi."""
    return Fraction(HALF_PARAM_BYTES + HALF_GRAD_BYTES + k) * psi


def zero1(psi, nd, k=K_ADAM_MIXED):
    """P_os: optimizer state partitioned: (2 + 2) Psi + K Psi / N_d."""
    return Fraction(HALF_PARAM_BYTES + HALF_GRAD_BYTES) * psi + Fraction(k * psi, nd)


def zero2(psi, nd, k=K_ADAM_MIXED):
    """P_os+g: optimizer state and gradients partitioned: 2 Psi + (2 + K) Psi / N_d."""
    return Fraction(HALF_PARAM_BYTES) * psi + Fraction((HALF_GRAD_BYTES + k) * psi, nd)


def zero3(psi, nd, k=K_ADAM_MIXED):
    """P_os+g+p: everything partitioned: (2 + 2 + K) Psi / N_d."""
    return Fraction((HALF_PARAM_BYTES + HALF_GRAD_BYTES + k) * psi, nd)


def optional_fp32_grads(psi, nd=1):
    """The optional fp32 gradient copy used when accumulating in fp32: 4 Psi,
    of which ZeRO-2 keeps 1/N_d ("DeepSpeed ZeRO", ZeRO Stage 2)."""
    return Fraction(4 * psi, nd)
