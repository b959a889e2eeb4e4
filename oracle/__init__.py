"""fp64 CPU oracle for the MatrixFSDP owner-local optimizer step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import or run anything in this package; the
product path (the CUDA library and its Python binding) never does, and shares no
code with it.  Everything here is plain, slow and written to be checked against
the paper by eye: NumPy in float64, library matmul as the only primitive, no
blocking, fusion or reordering.

Source: MatrixFSDP: Communication-Free Matrix Optimizers Under ZeRO-3 Parameter
Sharding (Gao, Xu, Zhang; arXiv 2607.05895) -- Abstract, Section 1 Introduction
and the FAQ on the paper's docshare page.  Where those pages are silent the
plainest reading is taken; each such reading is named in the function that
takes it.

Pins (tests/test_oracle_*.py check every function against something other than
itself): Newton-Schulz against its SVD closed form, the scalar quintic, special
cases and invariances; momentum against its closed forms at steps 1 and 2;
AdamW against its closed-form first step and torch.optim.AdamW; the planner
against brute force, Graham's LPT bound and a hand-worked layout.
"""
from .planner import plan_owners_ref, heaviest_rank_ref  # noqa: F401
from .muon import (bf16_bits_to_f64, momentum_ref, newton_schulz_ref,  # noqa: F401
                   muon_owner_step_ref, muon_matrix_ref, muon_scale_ref, muon_apply_ref)
from .adamw import adamw_ref  # noqa: F401
from .segments import (model_layout_ref, placement_segments_ref, segment_reduce_ref,  # noqa: F401
                       segment_gather_ref)
