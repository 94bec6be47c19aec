"""Routing of token-expert pairs (oracle side).

Test infrastructure only (see the package docstring).

Follows ``fp8_grouped_mm_experts_forward`` (source excerpt on the error page
"grouped_mm experts dispatch does not support activation_scheme='static'"): the S = T*K pairs are flattened in (token, k) order
(``top_k_index.reshape(-1)``), sorted by expert id (``torch.sort``) and the
hidden row of slot s is gathered by ``s // K``. The source excerpt of
``deepgemm_fp8_fp4_experts_forward`` (error record "DeepGEMM experts selected
on a model spanning multiple CUDA devices") adds a ``sorted_to_padded`` map:
each expert's rows start at an aligned offset of a padded grouped buffer. The
Mega MoE forward docstring (source excerpt of the error record "DeepGEMM Mega
MoE requires a process_group for the EP group") states that ids are global
and -1 marks a skipped slot.

Readings where the pages are silent:
* the sort is stable (equal ids keep ascending slot order) and a skipped slot
  gets the key E, so it sorts after every expert and joins no group;
* an id outside [-1, E) is invalid: it is treated as skipped and reported;
* the group alignment A is a parameter; padding rows belong to no slot.
"""
import numpy as np


def route(topk_idx, num_experts, align):
    """Stable counting sort of the flattened pairs plus the padded layout.

    Returns a dict of int64 arrays:
      keys            [S]    expert id per slot, E for skipped/invalid slots
      counts          [E]    pairs per expert
      offsets         [E+1]  exclusive scan of counts (unpadded sorted order)
      perm            [S]    sorted position -> slot (skipped slots last)
      padded_offsets  [E+1]  start row of each expert group, multiple of A
      inv             [S]    slot -> padded row, -1 for skipped slots
      row_slot        [M]    padded row -> slot, -1 for padding rows
      n_invalid              number of ids outside [-1, E)
    """
    idx = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    E = int(num_experts)
    S = idx.size
    invalid = (idx < -1) | (idx >= E)
    keys = np.where((idx < 0) | invalid, E, idx)
    counts = np.bincount(keys, minlength=E + 1)[:E]
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(keys, kind="stable")
    padded = (counts + align - 1) // align * align
    padded_offsets = np.zeros(E + 1, dtype=np.int64)
    padded_offsets[1:] = np.cumsum(padded)
    inv = np.full(S, -1, dtype=np.int64)
    M = int(padded_offsets[E])
    row_slot = np.full(M, -1, dtype=np.int64)
    for pos in range(int(offsets[E])):
        s = perm[pos]
        e = keys[s]
        row = padded_offsets[e] + (pos - offsets[e])
        inv[s] = row
        row_slot[row] = s
    return dict(keys=keys, counts=counts, offsets=offsets, perm=perm,
                padded_offsets=padded_offsets, inv=inv, row_slot=row_slot,
                n_invalid=int(invalid.sum()))
