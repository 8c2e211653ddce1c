"""The oracle indexer over many queries in a process pool.  Test infrastructure:
only the tests call it.

The pool is started with ``spawn``: the calling process may hold a CUDA context,
and a process forked after one is created can hang.  The workspace shared by every
query (page table, index-K cache, sizes) is handed to each worker once; the tasks
carry only their queries."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import oracle

_SHARED: dict = {}


def _init(page_table, cache_arg, k_scale, page_size, block_tokens, topk, max_blocks):
    _SHARED.update(page_table=page_table, cache=cache_arg, k_scale=k_scale, page_size=page_size,
                   block_tokens=block_tokens, topk=topk, max_blocks=max_blocks)


def _rows(task):
    idx_q, kv_len, table_offset = task
    s = _SHARED
    return oracle.indexer(idx_q, kv_len, table_offset, s["page_table"], s["cache"], s["k_scale"],
                          s["page_size"], s["block_tokens"], s["topk"], s["max_blocks"])


def indexer_rows(w, idx, cache_arg, chunk: int = 64, workers: int | None = None):
    """(block scores, top-k ids) of the oracle indexer for queries idx of workload w,
    in the order of idx."""
    idx = np.asarray(idx)
    parts = [idx[i:i + chunk] for i in range(0, idx.size, chunk)]
    tasks = [(np.ascontiguousarray(w.idx_q[p]), np.ascontiguousarray(w.kv_len[p]),
              np.ascontiguousarray(w.table_offset[p])) for p in parts]
    workers = workers or max(1, min(16, os.cpu_count() or 1, len(tasks)))
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_init,
                  initargs=(w.page_table, cache_arg, w.k_scale, w.page_size, w.block_tokens, w.topk,
                            w.max_blocks)) as pool:
        outs = pool.map(_rows, tasks)
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])
