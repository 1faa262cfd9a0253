"""fp64 CPU oracle for exact attention: test infrastructure, not product code.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import anything under this directory.
"""
