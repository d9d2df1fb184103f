"""fp64 CPU oracle for top-k sparse flash attention (forward + backward).

Test infrastructure only: imported by tests/, __graft_entry__.smoke() and the
CPU-baseline leg of bench.py, never by the product library.
"""
from .sfa import Problem, make_problem, token_keys, token_terms, sfa_fwd, sfa_bwd  # noqa: F401
