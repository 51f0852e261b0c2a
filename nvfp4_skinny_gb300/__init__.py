"""GB300 (sm_103a) NVFP4 weight-only skinny projection: y = x . dequant(W)^T for 1..32 rows.

The computation runs in the CUDA library built from ``csrc/`` (C ABI in
``include/nvfp4_skinny.h``); ``binding`` is a thin ctypes layer over it with the
same function names.  ``synth`` holds the seeded synthetic input generators.
"""
from .binding import (  # noqa: F401
    NVFP4_ERR_ALIGN, NVFP4_ERR_ARG, NVFP4_ERR_CUDA, NVFP4_ERR_M_RANGE, NVFP4_ERR_NOMEM, NVFP4_ERR_SHAPE,
    NVFP4_ERR_TIMEOUT, NVFP4_MAX_M, NVFP4_OK, NVFP4_OUT_BF16, NVFP4_OUT_F32, Nvfp4Error, Plan,
    nvfp4_abi_version, nvfp4_e4m3_encode, nvfp4_pack_codes, nvfp4_plan_check, nvfp4_plan_create,
    nvfp4_plan_create_ex, nvfp4_plan_destroy, nvfp4_plan_get_info, nvfp4_skinny_linear, nvfp4_status_string,
    nvfp4_unpack_codes,
)
