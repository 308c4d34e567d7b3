"""GB300-native logit-space verification for speculative decoding.

Thin Python binding over the C ABI in ``include/asv.h`` (``libasv.so``, built
in-tree by :func:`build`).  Every step of the verification runs in the
library's CUDA kernels; this module only checks tensor shapes, allocates the
outputs with PyTorch and passes raw device pointers and the current CUDA
stream.  There is no CPU fallback: on a machine without the library or
without a CUDA device the calls raise.

Entry points (same names as the C ABI):
  asymspec_verify        AsymSpec CDA gate + delta-fusion ("AsymSpec: Context-Asymmetric
                         Speculative Decoding for Agentic LLMs", sec. 4.1-4.2)
  asymspec_verify_sweep  the same for every (beta, gamma) of a grid from one read (sec. 5)
  asymspec_sci_verify    AsymSpec and one E2-SCI window on the same tensors from one read
  asymspec_verify_host   AsymSpec on host buffers (copies in and out on the call's stream)
  rapid_verify           RAPID retrieval-augmented target verification ("RAPID: Long-Context
                         Inference with Retrieval-Augmented Speculative Decoding", Key designs 2-4)
  sci_verify             E2-SCI JSD test against an adaptive threshold ("E2-SCI: Elastic
                         Edge-Cloud Speculative Decoding via Credit Inertia", Key design 3)
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    ASV_BF16,
    ASV_F32,
    DELTA_A,
    DELTA_A_MINUS_B,
    DELTA_T_MINUS_B,
    ASV_MODE_ASYMSPEC,
    ASV_MODE_RAPID,
    ASV_MODE_SCI,
    ASV_MODE_SWEEP,
    ASV_MODE_ASYMSPEC_SCI,
    AsymSciOutput,
    SweepOutput,
    asymspec_sci_verify,
    asymspec_verify_sweep,
    REQ_BAD_DRAFT,
    REQ_NONFINITE,
    REQ_TIMEOUT,
    AsvError,
    AsymSpecOutput,
    RapidOutput,
    SciOutput,
    SciParams,
    SciStabilisers,
    TAIL_KEEP_P,
    TAIL_RENORMALISE_ALL,
    asymspec_verify,
    asymspec_verify_host,
    host_arena_bytes,
    library,
    library_path,
    query_plan,
    rapid_verify,
    sci_state_decode,
    sci_state_new,
    sci_verify,
    set_kernel,
    set_tuning,
    KERNEL_CLUSTER,
    KERNEL_DEFAULT,
    KERNEL_STAGED,
    workspace_bytes,
)
from .nvcc_build import build  # noqa: F401
