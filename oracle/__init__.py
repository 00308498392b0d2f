"""CPU oracle of the Clef JointSchemaHead forward pass (fp64 NumPy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or link
this package: only the tests, the smoke check of the entry module and the CPU
baseline leg of the benchmark use it.  It shares no code with the CUDA path.
"""
from .clef_head import (
    EPS_COS, EPS_LN, HeadParams, answers, cosine, cross_attention, field_aggregate,
    gelu, head_forward, joint_layer, layer_norm, memory_rows, option_query,
    pool_record, question_softmax, routing_layer, scorer_logits, self_attention,
    span_raw_sums,
)
