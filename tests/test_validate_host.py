"""Opt-in host validation of a call's index data (``smla_validate_host`` and
the binding's SMLA_VALIDATE=1 hook), on the CPU: the named workloads pass,
each rule reports its first bad entry by location, and on randomly planted bad
entries it fails exactly when the oracle (which raises on an index outside its
pool) does."""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_mla_decode_token_gb300 import binding as B
from sparse_mla_decode_token_gb300 import build as smla_build
from sparse_mla_decode_token_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def lib():
    smla_build.build()
    return B.lib()


def host_args(w, **over):
    """smla_args whose index-data pointers are numpy arrays of ``w`` (kept
    alive in the returned list); ``over`` replaces arrays by name."""
    arrays = dict(indices=w.indices, topk_lens=w.topk_lens, seq_lens=w.seq_lens, cum=w.cum_seq_lens_q,
                  bt=w.comp_block_tables, hca=w.hca_seq_lens, win=w.swa_topk_lens)
    arrays.update(over)
    keep = {k: None if v is None else np.ascontiguousarray(v, dtype=np.int32) for k, v in arrays.items()}

    def ptr(k):
        return None if keep[k] is None else keep[k].ctypes.data

    a = B.SmlaArgs()
    a.sum_q, a.batch, a.num_heads, a.width = w.sum_q, w.batch, w.num_heads, w.width
    a.dtype = B.SMLA_BF16 if w.dtype == "bf16" else B.SMLA_E4M3
    a.swa_rows, a.comp_rows = w.swa_kv.shape[0], w.comp_kv.shape[0]
    a.sparse_indices, a.indices_row_stride = ptr("indices"), keep["indices"].shape[1]
    a.sparse_topk_lens, a.seq_lens, a.cum_seq_lens_q = ptr("topk_lens"), ptr("seq_lens"), ptr("cum")
    a.swa_topk_lens = ptr("win")
    if keep["bt"] is not None:
        a.comp_block_tables, a.block_table_stride = ptr("bt"), keep["bt"].shape[1]
        a.comp_max_pages, a.comp_page_size, a.hca_seq_lens = keep["bt"].shape[1], w.comp_page_size, ptr("hca")
    return a, keep


def validate(w, **over):
    a, keep = host_args(w, **over)
    B.smla_validate_host(a)
    del keep


def small(seed=3, **kw):
    base = dict(name="v", seed=seed, dtype="bf16", batch=3, q_lens=[1, 3, 2], num_heads=64, swa_rows=3 * 130,
                comp_rows=300, width=128 + 40, seq_lens=[500, 700, 900], ring_len=130,
                topk_lens=[160, 168, 150, 140, 128, 167], sinks=False, varlen=True)
    base.update(kw)
    return W.make_workload(**base)


def paged(seed=4, **kw):
    base = dict(name="vp", seed=seed, dtype="bf16", batch=3, q_lens=[1, 2, 1], num_heads=64, swa_rows=3 * 130,
                comp_pages=16, page_size=8, max_pages=5, hca_seq_lens=[128 + 37, 128 + 8, 100],
                seq_lens=[5000, 60, 3000], ring_len=130, topk_lens=[160, 170, 140, 168],
                swa_topk_lens=[128, 17, 0, 64], varlen=True)
    base.update(kw)
    return W.make_paged_workload(**base)


@pytest.mark.parametrize("n", [1, 2, 4, 6])
def test_named_workloads_pass(n):
    validate(W.config_workload(n))


def test_small_workloads_pass():
    validate(small())
    validate(paged())


def expect(w, match, **over):
    with pytest.raises(B.SmlaError) as e:
        validate(w, **over)
    assert e.value.status == B.SMLA_ERR_INVALID_ARG
    assert match in str(e.value), str(e.value)


def test_index_form_rules():
    w = small()
    ind = w.indices.copy()
    ind[2, 130] = 300                                        # compressed pool has 300 rows
    expect(w, "token 2 (request 1) column 130: index 300 outside the compressed pool of 300 rows", indices=ind)
    ind = w.indices.copy()
    ind[4, 5] = -7
    expect(w, "token 4 (request 2) column 5: index -7 outside the SWA pool", indices=ind)
    # entries the kernels never read are not checked
    ind = w.indices.copy()
    ind[3, 145] = 10 ** 6                                    # token 3 reads columns < 140
    validate(w, indices=ind)
    ind = w.indices.copy()
    ind[0, 127] = 10 ** 6
    validate(w, indices=ind, seq_lens=np.array([100, 700, 900]))   # window of token 0 is 100 columns
    expect(w, "column 127: index 1000000 outside the SWA pool", indices=ind)


def test_request_bookkeeping_rules():
    w = small()
    expect(w, "cum_seq_lens_q[0] = 1, not 0", cum=np.array([1, 1, 4, 6]))
    expect(w, "cum_seq_lens_q gives request 2 a negative length (4 -> 3)", cum=np.array([0, 1, 4, 3]))
    expect(w, "cum_seq_lens_q[3] = 5, not sum_q = 6", cum=np.array([0, 1, 4, 5]))


def test_lengths_are_clamped_as_the_kernels_clamp_them():
    """Lengths outside their range are clamped by the contract, not errors;
    the clamped range decides which entries are checked."""
    w = small()
    ind = w.indices.copy()
    ind[0, 165] = 10 ** 6                                    # token 0 reads columns < 160 ...
    validate(w, indices=ind)
    expect(w, "token 0 (request 0) column 165", indices=ind,
           topk_lens=np.array([10 ** 6, 168, 150, 140, 128, 167]))   # ... unless its length clamps to 168
    validate(w, indices=ind, topk_lens=np.array([-5, 168, 150, 140, 128, 167]))   # clamps to 0: nothing read
    ind = w.indices.copy()
    ind[2, 100] = 10 ** 6
    validate(w, indices=ind, win=np.array([0, 0, -3, 0, 0, 0]))       # window clamps to 0
    expect(w, "token 2 (request 1) column 100", indices=ind, win=np.array([0, 0, 500, 0, 0, 0]))
    validate(w, indices=ind, seq_lens=np.array([500, 1, 900]))        # position < 0: empty window


def test_page_table_rules():
    w = paged()
    bt = w.comp_block_tables.copy()
    bt[0, 2] = -1                                            # inside token 0's 37-slot footprint
    expect(w, "token 0 (request 0) compressed slot 16: page -1 (table column 2) gives row -8", bt=bt)
    bt = w.comp_block_tables.copy()
    bt[1, 0] = 16                                            # 16 pages of 8 rows: page 16 starts at row 128
    expect(w, "token 1 (request 1) compressed slot 0: page 16 (table column 0) gives row 128", bt=bt)
    bt = w.comp_block_tables.copy()
    bt[1, 3] = 10 ** 6                                       # past request 1's one-page footprint: never read
    validate(w, bt=bt)
    bt[1, [1, 2, 4]] = [1, 2, 4]                             # a 40-slot footprint reads all five pages
    expect(w, "token 1 (request 1) compressed slot 24: page 1000000 (table column 3)", bt=bt,
           hca=np.array([165, 168, 100]))


@pytest.mark.parametrize("seed", range(12))
def test_agrees_with_the_oracle_on_planted_entries(seed):
    """A random bad index or page somewhere in the table: the validator fails
    exactly when the oracle raises on some token (an entry the token reads)."""
    rng = np.random.default_rng(seed)
    w = paged(seed=seed) if seed % 2 else small(seed=seed)
    over = {}
    if w.comp_block_tables is not None and rng.random() < 0.5:
        bt = w.comp_block_tables.copy()
        t, c = rng.integers(bt.shape[0]), rng.integers(bt.shape[1])
        bt[t, c] = rng.choice([-1, 16, 10 ** 5])
        over["bt"] = bt
    else:
        ind = w.indices.copy()
        t, j = rng.integers(ind.shape[0]), rng.integers(ind.shape[1])
        ind[t, j] = rng.choice([-2, 10 ** 6])
        over["indices"] = ind
    oracle_raises = False
    for tok in range(w.sum_q):
        try:
            orc.valid_slots(tok, indices=over.get("indices", w.indices), topk_lens=w.topk_lens,
                            seq_lens=w.seq_lens, cum_seq_lens_q=w.cum_seq_lens_q, batch=w.batch,
                            swa_rows=w.swa_kv.shape[0], comp_rows=w.comp_kv.shape[0], width=w.width,
                            swa_topk_lens=w.swa_topk_lens, comp_block_tables=over.get("bt", w.comp_block_tables),
                            comp_page_size=w.comp_page_size, hca_seq_lens=w.hca_seq_lens)
        except IndexError:
            oracle_raises = True
    a, keep = host_args(w, **over)
    status = B.lib().smla_validate_host(ctypes.byref(a))
    assert (status == B.SMLA_ERR_INVALID_ARG) == oracle_raises, (seed, B.smla_last_error())


def test_binding_hook_runs_only_when_enabled(monkeypatch):
    """SMLA_VALIDATE=1 makes make_args validate host copies of the index data
    (here host tensors, so a good call then stops at the device check)."""
    w = small()
    ind = w.indices.copy()
    ind[2, 130] = 300
    kw = dict(q=torch.zeros(w.sum_q, 64, 512, dtype=torch.bfloat16),
              swa_kv=torch.zeros(390, 512, dtype=torch.bfloat16),
              compressed_kv=torch.zeros(300, 512, dtype=torch.bfloat16),
              sparse_indices=torch.from_numpy(ind), seq_lens=torch.from_numpy(w.seq_lens.astype(np.int32)),
              out=torch.empty(w.sum_q, 64, 512, dtype=torch.bfloat16),
              sparse_topk_lens=torch.from_numpy(w.topk_lens.astype(np.int32)),
              cum_seq_lens_q=torch.from_numpy(w.cum_seq_lens_q.astype(np.int32)))
    monkeypatch.delenv("SMLA_VALIDATE", raising=False)
    with pytest.raises(ValueError, match="CUDA device"):
        B.make_args(**kw)
    monkeypatch.setenv("SMLA_VALIDATE", "1")
    with pytest.raises(B.SmlaError, match="column 130: index 300"):
        B.make_args(**kw)
    kw["sparse_indices"] = torch.from_numpy(w.indices)
    with pytest.raises(ValueError, match="CUDA device"):
        B.make_args(**kw)
