"""GB300 CVR scoring library: a C-ABI shared library (libcvr.so, include/cvr.h) of hand-written
sm_103a CUDA kernels for the HyFormer-style CVR ranking forward pass, with a thin ctypes binding."""
from .binding import (NOALLOC_MAX_CAND, OPT_ATTENTION_TC, OPT_CUDA_GRAPH, OPT_KEEP_STAGES, OPT_PDL, OPT_PLE_INT8, OPT_PROFILE, STAGE_EXPERTS, STAGE_GATES, STAGE_H, STAGE_Q, STAGE_Y, STAGE_Z,
                      Config, CvrError, Scorer, Weights, lib, make_config, make_weights)
from ._build import build

__all__ = ["Config", "Weights", "Scorer", "CvrError", "lib", "make_config", "make_weights", "build", "OPT_PROFILE",
           "OPT_CUDA_GRAPH", "OPT_PDL", "OPT_ATTENTION_TC", "OPT_PLE_INT8", "OPT_KEEP_STAGES", "NOALLOC_MAX_CAND", "STAGE_H", "STAGE_Z", "STAGE_Q", "STAGE_Y", "STAGE_EXPERTS", "STAGE_GATES"]
