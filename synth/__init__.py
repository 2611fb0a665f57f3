"""Seeded synthetic inputs: model artifacts and prompts.

This module is the one piece shared by the CPU oracle's tests and the CUDA
path. It holds none of the integer method's arithmetic: it only draws seeded
random weights, scales and prompts, and it stands in for the float,
offline preparation stage (calibration and table building) that the DetLLM
README ("Layout": prepare.py, float -> int artifact) keeps outside the
integer forward pass. Everything it computes in float64 is written once
into the artifact file and from then on read as data by both sides.

Weight distributions follow the workloads the pages run: int8 weights
round(N(0, 24)) clipped to +-127, per-output-channel dyadic scales with a
mantissa uniform in [2^14, 2^15) and shift 22, int16 RMSNorm gammas uniform
in [2^11, 2^13), RoPE tables in int16 Q14 built in float64.
"""
from .artifact import (MODEL_SHAPES, ModelShape, write_artifact, artifact_path,
                       read_header, ensure_artifact)
from .prompts import prompt_ids, coprompt_lengths

__all__ = ["MODEL_SHAPES", "ModelShape", "write_artifact", "artifact_path",
           "read_header", "ensure_artifact", "prompt_ids", "coprompt_lengths"]
