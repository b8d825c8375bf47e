"""libsinkattn: grouped-query attention with a per-head learned sink, for GB300 (sm_103a).

``gqa_attention_learned_head_gb300.sinkattn`` is the Python binding of the C
library (``include/sinkattn.h``); ``workloads`` draws seeded synthetic inputs.
The binding is imported lazily so that the input generators stay usable on a
machine where the CUDA library has not been built.
"""
__all__ = ["sinkattn", "workloads"]
