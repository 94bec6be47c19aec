"""Slow, plain fp64 CPU oracle for the block-scaled MoE experts forward.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
package: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it. It shares no code, table or constant with the CUDA
library in ``block_scaled_moe_expert_gb300/``; both sides only consume the
same seeded input bytes.

Sources. The method is spread over a handful of transformers pages:

* ``fp8_grouped_mm_experts_forward`` (source excerpt on the error page
  "grouped_mm experts dispatch does not support activation_scheme='static'"): flatten the top-k pairs, sort them by expert, gather rows by
  ``perm // K``; afterwards zero the sentinel rows and reduce the top-k rows
  per token with a deterministic reshape+sum, then cast to the input dtype.
  The same page states that the grouped dispatch quantizes activations
  dynamically per block.
* "deepgemm_fp8_fp4_experts_forward" (source excerpt of the error record
  "DeepGEMM experts selected on a model spanning multiple CUDA devices"): the
  sorted-to-padded grouped layout, the grouped FP8 x FP8/FP4 matmul, and the
  bf16-only / static-scheme / multi-device refusals.
* "DeepGEMM Mega MoE" forward docstring (source excerpt of the error record
  "DeepGEMM Mega MoE requires a process_group for the EP group"): top-k ids are global expert ids with -1 marking skipped slots;
  gate_up and down weights carry UE8M0 scale factors; ``swiglu_limit`` is an
  optional clamp, unclamped when absent.

Exact number formats (e4m3, e2m1, UE8M0), the 1x128 power-of-two activation
rule and the 128x128 / 1x32 weight blockings are fixed by the workload
definitions that accompany those pages; the readings taken where the pages
are silent are listed in each module.

Modules:
  formats  -- exact decode tables and the activation quantizers (e4m3 1x128;
              e2m1 1x32 for the FP4-activation variant).
  routing  -- flatten + stable counting sort + padded grouped layout.
  moe      -- the experts forward itself (per pair, fp64).
"""
