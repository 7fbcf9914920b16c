"""GB300-native KV-cache token eviction.

Five operations, each one call into ``libkvc.so`` (hand-written CUDA for sm_103a):

* ``kv_score_obs``     observation-window Q.K^T, softmax, per-head column mass;
* ``hubkv_refine``     local hubs (width-5 max-pool), gamma discount, clipped head
                       weight, r^2 ratio gate;
* ``kv_select_topk``   budgeted per-head Top-K with a protected recent window;
* ``kv_compact``       gather of the kept K/V rows into a slot cache;
* ``h2o_decode_step``  decode attention with accumulated scores and at most one
                       eviction per KV head.

The binding (``kv_cache_compression_obs_gb300.api``) only marshals arguments;
importing it loads the CUDA library and raises if it is missing.  ``gen`` and
``configs`` are plain Python and do not load the library.
"""
from .configs import ALL, BY_NAME, Workload  # noqa: F401

_API_NAMES = {"kv_score_obs", "hubkv_refine", "kv_select_topk", "kv_compact",
              "h2o_decode_step", "kv_workspace_size", "KvcError", "compress_prefill",
              "compress_prefill_host", "kv_select_budget", "kv_compact_ragged", "kv_score_nested"}


def __getattr__(name):
    if name in _API_NAMES:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
