"""GB300 (sm_103a) library for the hot path of speculative decoding with
n-gram drafts: device bigram/trigram tables (``ngram_update``,
``ngram_draft``), a single-pass Leviathan/Chen verifier with Gumbel-max
residual / bonus sampling, kv_len rollback and an EMA gate
(``spec_verify``), the history append (``spec_append``), and the
decode-step bookkeeping around them: a KV block pool (``KvPool``) and a
device step counter (``step_advance``) for steps replayed from a CUDA graph.

The compute runs in hand-written CUDA kernels behind the C ABI of
``include/specng.h`` (``libspecng.so``); this package is the thin binding.
"""
from .capi import (  # noqa: F401
    KvPool,
    NgramTable,
    SpecngError,
    VerifyParams,
    get_counters,
    get_status,
    lib_path,
    load,
    ngram_draft,
    ngram_update,
    philox4x32_10,
    set_verify_marker,
    spec_append,
    spec_commit,
    spec_verify,
    spec_verify_lmhead,
    spec_verify_lmhead_workspace,
    spec_verify_lmhead_workspace_bytes,
    spec_verify_noalloc,
    spec_verify_workspace,
    spec_verify_workspace_bytes,
    status_names,
    step_advance,
)
