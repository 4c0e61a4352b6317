"""CPU oracle for the InfiniGen decode hot path (test infrastructure only; see infinigen.py)."""
