"""float64 CPU oracle for the MuonH step: test infrastructure only (see muonh.py)."""
