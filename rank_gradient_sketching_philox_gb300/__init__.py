"""GB300 (sm_103a) library for randomized low-rank gradient sketching of linear
layers (RGC / LoGRA): seeded projections, projected inputs, fp32 sketch
accumulation and the fused rebuild + stochastically rounded BF16 update.

The compute path is the C-ABI shared library ``lib/libsketch.so`` (declared in
``include/sketch.h``); ``binding`` is its thin Python wrapper.
"""
from .binding import (PROJ_GAUSSIAN_QR, PROJ_RADEMACHER, SketchError, accumulate,  # noqa: F401
                      accumulate_batched, accumulate_fp32xp_batched, apply_update_normsgd,
                      apply_update_normsgd_batched, apply_update_sgd, apply_update_sgd_batched,
                      kernel_launches, project_inputs, project_inputs_batched,
                      project_inputs_fp32xp_batched, project_inputs_grouped_batched,
                      projection_split_elems, read_device_errors, read_exact_count, sample_projection,
                      sample_projection_batched, split_projection_batched, split_projection_grouped,
                      workspace_bytes, workspace_bytes_batched, xp_split_cols)
