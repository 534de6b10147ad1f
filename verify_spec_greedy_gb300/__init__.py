"""libmtpspec: the data-parallel hot path of MTP speculative decoding on GB300 (sm_103a).

The computation is in the CUDA library built from ``csrc/`` (see ``build.py``); this
package only loads it and marshals arguments.  ``inputs`` holds the seeded synthetic
workloads used by the tests and the benchmark.
"""
from ._binding import (  # noqa: F401
    BF16, F32, LIB_PATH, STATUS_BAD_DRAFT_ID, STATUS_BAD_PARAM, STATUS_TIMEOUT, MtpSpecError,
    load, mtpspec_launch_count, mtpspec_selftest_wait_timeout, mtp_draft_input,
    mtp_draft_input_workspace_bytes, mtp_greedy_draft,
    mtp_draft_steps, mtp_draft_steps_workspace_bytes, mtp_lm_head_greedy,
    mtp_lm_head_greedy_workspace_bytes, mtp_lm_head_topk, mtp_lm_head_topk_workspace_bytes,
    mtp_state_fixup, mtp_state_snapshot,
    spec_verify_greedy,
    spec_verify_sample, spec_verify_sample_static, spec_verify_workspace_bytes,
    status_string)
