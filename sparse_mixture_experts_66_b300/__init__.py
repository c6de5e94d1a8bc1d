"""Sparse Mixture-of-Experts layer forward for B300 (sm_103a).

The compute lives in ``libmoe.so`` (CUDA kernels behind the C ABI of
``include/moe.h``); :mod:`.moe` is its thin ctypes binding and
:mod:`.workload` draws the seeded synthetic inputs.
"""
from . import moe, workload  # noqa: F401
from .moe import (MoeConfig, MoeError, Workspace, config_of, forward, make_config, moe_capacity,  # noqa: F401
                  moe_combine, moe_dispatch, moe_expert_ffn, moe_forward, moe_get_device_status,
                  moe_get_workspace_layout, moe_route, moe_workspace_bytes, moe_workspace_init)
