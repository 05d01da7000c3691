"""CPU fp64 oracle (test infrastructure only; see ``kd_oracle``)."""
from .kd_oracle import (  # noqa: F401
    dense_teacher_grid,
    kd_backward,
    kd_backward_shard,
    kd_forward,
    kd_forward_shard,
    kd_from_logits,
    logsumexp_rows,
    mean_loss,
    student_logits,
    teacher_log_probs,
    teacher_topk,
)
