"""GB300-native MuonClip optimizer step: per-head max-logit scan, QK-Clip
(MHA / MLA / global) and the Muon update with quintic Newton-Schulz, as a
C-ABI CUDA library for sm_103a (``include/mc_max.h``) with this thin
ctypes binding.  See ``api`` for the functions and ``step`` for the composed
MuonClip step."""
from .api import *  # noqa: F401,F403
from .api import __all__ as _api_all
from .step import CapturedStep, muonclip_step_mha, muonclip_step_mla  # noqa: F401

__all__ = list(_api_all) + ["CapturedStep", "muonclip_step_mha", "muonclip_step_mla"]
